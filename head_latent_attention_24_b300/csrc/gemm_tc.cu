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
// accumulator D[m][n] lives in TMEM.
//
// A stage holds CPB (1, 2 or 4) column chunks of 64: the weight tile arrives
// as one TMA box through a 4-D view {64 columns, rows, column chunks, batch}
// with the chunk outside the row, which lands chunk-major in the 128-byte
// swizzled K-major layout tcgen05 reads, and the activation chunks as a second
// box. An SM completes only about two million TMA copies per second whatever
// their size, so large boxes are what lets the weights stream at HBM speed.
//
// To spread a weight matrix over the SMs the reduction is split along K
// across the CTAs of a thread-block cluster (up to 8); each CTA writes its
// partial tile to its own shared memory and the cluster sums the partials in
// a fixed order through distributed shared memory, so results do not depend
// on timing. When there are more 128-row tiles than SMs (W_UK^T, batched over
// heads), one CTA instead computes MT tiles that share their activations.
//
// Warp roles: warp 0 issues TMA, warp 1 owns TMEM and issues tcgen05.mma from
// one thread, warps 2-5 drain TMEM, reduce and run the epilogue. Every
// mbarrier wait is bounded; on expiry the CTA records MLA_DEV_TIMEOUT and
// skips the rest of its work (still joining the cluster barriers).
#include <mutex>
#include <vector>

#include "internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int BM = 128;            // weight rows per tile (MMA M)
constexpr int BK = 64;             // reduction columns per chunk (128 B of bf16)
constexpr int CHUNK_A = BM * BK * 2;   // 16 KB: one chunk of a weight tile
// Row stride (floats) of the fp32 partial tiles in shared memory: the store
// loop reads 8 consecutive rows m of two activation rows n per warp, and the
// 4-float pad puts those two rows on different banks.
constexpr int CS_LD = BM + 4;
constexpr int NTHREADS = 192;
constexpr int MAX_SPLITS = 8;
constexpr int MAX_MT = 4;
constexpr int SMEM_ONE = 200 * 1024;   // stage budget with one CTA per SM
constexpr int SMEM_TWO = 100 * 1024;   // with two
constexpr long long WAIT_CYCLES = 4000000000LL;  // ~2 s

struct Params {
  int mstart[4];               // first tile of each segment; mstart[nseg] = all tiles
  int mtiles_total;
  int mt;                      // 128-row tiles per CTA (> 1 only without split-K)
  int rows[3], col0[3];
  int N, K, Z;
  int n_tile, nstage, stage_bytes, splits, kstages;
  uint32_t tmem_cols, idesc;
  int epi[3]; void* out[3]; long long ldo[3], bo[3];
  long long seg_stride[3]; int seg_off[3]; int seg_len[3];
  const float* rope_cos; const float* rope_sin; int d_r; int max_pos;
  const int32_t* pos;
  const int32_t* tok_seq; const int32_t* tok_pos; int cache_batch; int max_len; int d_c; int row_width;
  // > 0: the epilogue first copies, for the tile's activation rows, their
  // positions (and cache sequences) and the RoPE cos/sin rows at those
  // positions into shared memory at this offset (layout in stage_rope).
  int rope_off;
  int32_t* status;
};

struct Ctl {
  uint64_t full[8], empty[8], acc_full;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Ctl& ctl, int32_t* status) {
  if (*reinterpret_cast<volatile int*>(&ctl.abort)) return false;
  if (mbar_wait(bar, parity, WAIT_CYCLES)) return true;
  atomicOr(status, MLA_DEV_TIMEOUT);
  *reinterpret_cast<volatile int*>(&ctl.abort) = 1;
  return false;
}

__device__ __forceinline__ float rope_apply(float v, float partner, bool first_half, float c, float s) {
  return first_half ? (v * c - partner * s) : (v * c + partner * s);
}

// RoPE on 8 consecutive rows; the partner rows, cos and sin come as pairs of
// 16-byte loads (each pointer starts an 8-row group, d_r / 2 is a multiple
// of 8, and every row of the tables and partial tiles is 16-byte aligned).
__device__ __forceinline__ void rope8(float (&v)[8], const float* pr, bool first, const float* tc, const float* ts) {
  float q[8], c[8], sn[8];
  *reinterpret_cast<float4*>(q) = *reinterpret_cast<const float4*>(pr);
  *reinterpret_cast<float4*>(q + 4) = *reinterpret_cast<const float4*>(pr + 4);
  *reinterpret_cast<float4*>(c) = *reinterpret_cast<const float4*>(tc);
  *reinterpret_cast<float4*>(c + 4) = *reinterpret_cast<const float4*>(tc + 4);
  *reinterpret_cast<float4*>(sn) = *reinterpret_cast<const float4*>(ts);
  *reinterpret_cast<float4*>(sn + 4) = *reinterpret_cast<const float4*>(ts + 4);
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = rope_apply(v[e], q[e], first, c[e], sn[e]);
}

// Shared-memory copy of what the RoPE and cache-row epilogues read per
// activation row n of the tile: rc[n][j], rs[n][j] (cos, sin at the row's
// position, j < d_r/2), then pos_s[n] and seq_s[n] as stored (range checks
// stay with the epilogue). The 128 epilogue threads fill it with independent
// loads while the MMAs run, so the store loop reads no global memory.
__device__ __forceinline__ void stage_rope(const Params& p, uint8_t* smem, int n0, int n_valid, bool append, int et) {
  const int half = p.d_r / 2;
  float* rc = reinterpret_cast<float*>(smem + p.rope_off);
  float* rs = rc + p.n_tile * half;
  int32_t* pos_s = reinterpret_cast<int32_t*>(rs + p.n_tile * half);
  int32_t* seq_s = pos_s + p.n_tile;
  const int32_t* pos = append ? p.tok_pos : p.pos;
  for (int n = et; n < n_valid; n += 128) {
    pos_s[n] = pos[n0 + n];
    seq_s[n] = append ? (p.tok_seq ? p.tok_seq[n0 + n] : n0 + n) : 0;
  }
  for (int i = et; i < n_valid * half; i += 128) {
    const int n = i / half, j = i - n * half;
    int ps = pos[n0 + n];
    ps = ps < 0 ? 0 : (ps >= p.max_pos ? p.max_pos - 1 : ps);
    rc[i] = p.rope_cos[(long long)ps * half + j];
    rs[i] = p.rope_sin[(long long)ps * half + j];
  }
}

// CPB: column chunks per stage. TRANS: the weights are stored [K rows][M
// columns] and read MN-major (A'[m, k] = W[k, m]).
template <int CPB, bool TRANS>
__global__ void __launch_bounds__(NTHREADS, 2)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
                   const __grid_constant__ CUtensorMap map_w2, const __grid_constant__ CUtensorMap map_x,
                   const Params p) {
  constexpr int A_TILE = CPB * CHUNK_A;   // one weight tile of one stage
  constexpr int KSTEPS = CPB * (BK / 16);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Ctl ctl;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.splits, MT = p.mt;
  const int group = blockIdx.x / S, split = blockIdx.x % S;
  const int tile0 = group * MT;
  const int seg = (tile0 >= p.mstart[1] ? 1 : 0) + (tile0 >= p.mstart[2] ? 1 : 0);
  const int m0 = (tile0 - p.mstart[seg]) * BM;
  const int n0 = blockIdx.y * p.n_tile;
  const int z = blockIdx.z;
  const int ks0 = (int)((long long)split * p.kstages / S), ks1 = (int)((long long)(split + 1) * p.kstages / S);
  const int nk = ks1 - ks0;
  const CUtensorMap* map_w = seg == 0 ? &map_w0 : (seg == 1 ? &map_w1 : &map_w2);

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.nstage; ++i) { mbar_init(&ctl.full[i], 1); mbar_init(&ctl.empty[i], 1); }
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
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(map_w);
      prefetch_tensormap(&map_x);
      const uint32_t bytes = (uint32_t)p.stage_bytes;
      auto load_w = [&](int i) {
        const int st = i % p.nstage;
        uint8_t* sa = smem + st * p.stage_bytes;
        const int kc = (ks0 + i) * CPB;   // first column chunk of the stage
        for (int t = 0; t < MT; ++t) {
          if (TRANS) tma_load_4d(sa + t * A_TILE, map_w, &ctl.full[st], 0, kc * BK, (m0 + t * BM) / 64, z);
          else tma_load_4d(sa + t * A_TILE, map_w, &ctl.full[st], 0, m0 + t * BM, kc, z);
        }
      };
      auto load_x = [&](int i) {
        const int st = i % p.nstage;
        tma_load_4d(smem + st * p.stage_bytes + MT * A_TILE, &map_x, &ctl.full[st], 0, n0, (ks0 + i) * CPB, z);
      };
      // The weights of the first stages are read-only inputs: they stream in
      // while the previous kernel finishes; the activations wait for it.
      const int pre = nk < p.nstage ? nk : p.nstage;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&ctl.full[i], bytes);
        load_w(i);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) load_x(i);
      int issued = pre;
      for (int i = pre; i < nk; ++i) {
        const int st = i % p.nstage;
        if (!wait_bar(&ctl.empty[st], ((i / p.nstage) - 1) & 1, ctl, p.status)) break;
        mbar_arrive_expect_tx(&ctl.full[st], bytes);
        load_w(i);
        load_x(i);
        issued = i + 1;
      }
      if (issued < nk) {
        // Aborted: wait (bounded) until every stage loaded so far has landed,
        // before the epilogue reuses the stage buffers or the CTA exits. The
        // last load into stage s filled its phase (last / nstage).
        for (int st = 0; st < p.nstage && st < issued; ++st) {
          const int last = st + p.nstage * ((issued - 1 - st) / p.nstage);
          mbar_wait(&ctl.full[st], (uint32_t)((last / p.nstage) & 1), WAIT_CYCLES / 8);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Descriptors are built once; each MMA adds a byte offset / 16 to the
      // start-address field (shared addresses stay below 256 KB).
      const uint32_t sbase = smem_u32(smem);
      const uint64_t a_desc0 = TRANS ? sdesc_sw128(sbase, CPB * BK * 128, 1024) : sdesc_sw128(sbase, 16, 1024);
      const uint64_t x_desc0 = sdesc_sw128(sbase, 16, 1024);
      const uint32_t x_chunk = (uint32_t)p.n_tile * 128;
      for (int i = 0; i < nk; ++i) {
        const int st = i % p.nstage;
        if (!wait_bar(&ctl.full[st], (i / p.nstage) & 1, ctl, p.status)) break;
        tc_fence_after();
        const uint32_t soff = (uint32_t)(st * p.stage_bytes);
        const uint64_t xd = x_desc0 + ((soff + (uint32_t)MT * A_TILE) >> 4);
        for (int t = 0; t < MT; ++t) {
          const uint64_t ad = a_desc0 + ((soff + (uint32_t)t * A_TILE) >> 4);
          const uint32_t d = tbase + (uint32_t)(t * p.n_tile);
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            const uint32_t a_off = TRANS ? (uint32_t)(kk * 2048) : (uint32_t)((kk >> 2) * CHUNK_A + (kk & 3) * 32);
            const uint64_t xk = xd + (((uint32_t)(kk >> 2) * x_chunk + (uint32_t)(kk & 3) * 32) >> 4);
            mma_bf16(d, ad + (a_off >> 4), xk, p.idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&ctl.empty[st]);
      }
      mma_commit(&ctl.acc_full);
      // no MMA of this CTA is still running when it frees its TMEM
      mbar_wait(&ctl.acc_full, 0, WAIT_CYCLES / 8);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps 2..5
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;           // this thread's TMEM lane = tile row
    float* cs = reinterpret_cast<float*>(smem);  // [MT][n_tile][CS_LD] partials, reuses the stages
    pdl_wait();   // before the epilogue reads indices or writes the output
    if (p.rope_off) {
      bool append = false;
      for (int sg = 0; sg < 3; ++sg) append = append || p.epi[sg] == EPI_APPEND;
      stage_rope(p, smem, n0, min(p.n_tile, p.N - n0), append, threadIdx.x - 64);
      asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
    }
    // warp-uniform: the TMEM loads below are warp-collective
    const bool ok = __all_sync(0xffffffffu, nk > 0 && wait_bar(&ctl.acc_full, 0, ctl, p.status));
    if (ok) tc_fence_after();
    // After an abort the stage buffers may still be receiving loads (the
    // producer drains them before the cluster barrier below): leave them
    // alone; the result is void and the status word says so.
    for (int t = 0; t < MT && ok; ++t) {
      for (int c = 0; c < p.n_tile; c += 64) {
        float v[64];
        const int nc = min(64, p.n_tile - c);   // n_tile is a multiple of 16
        {
          const uint32_t ta = tbase + (static_cast<uint32_t>(quarter * 32) << 16) + (uint32_t)(t * p.n_tile + c);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (16 * q < nc) tmem_ld16(ta + 16 * q, *reinterpret_cast<float(*)[16]>(v + 16 * q));
          tmem_ld_wait();
        }
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i < nc) cs[(t * p.n_tile + c + i) * CS_LD + m] = v[i];
      }
    }
  }

  // ---------------------------------------------------------------- split-K sum
  __syncwarp();
  tc_fence_before();
  cluster_sync();  // every partial tile of the cluster is in shared memory
  const int n_valid = min(p.n_tile, p.N - n0);
  if (warp >= 2 && S > 1) {
    // MT == 1 whenever S > 1. Each warp sums rows n of the tile (this CTA's
    // rows n = split + S j) over the S partials, in split order; the loads of
    // two rows from all S CTAs are issued before any of them is used.
    const int et = threadIdx.x - 64;
    float* cs = reinterpret_cast<float*>(smem);
    const uint32_t cs_addr = smem_u32(cs);
    const int rgrp = et >> 5, m4 = (et & 31) * 4;
    for (int nb = split + S * rgrp; nb < n_valid; nb += 8 * S) {
      float4 v[2][MAX_SPLITS];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int n = nb + q * 4 * S;
#pragma unroll
        for (int r = 0; r < MAX_SPLITS; ++r)
          if (r < S && n < n_valid) {
            const uint32_t a = mapa_shared(cs_addr + (uint32_t)((n * CS_LD + m4) * 4), (uint32_t)r);
            asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                         : "=f"(v[q][r].x), "=f"(v[q][r].y), "=f"(v[q][r].z), "=f"(v[q][r].w)
                         : "r"(a));
          }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int n = nb + q * 4 * S;
        if (n >= n_valid) continue;
        float4 acc = v[q][0];
#pragma unroll
        for (int r = 1; r < MAX_SPLITS; ++r)
          if (r < S) { acc.x += v[q][r].x; acc.y += v[q][r].y; acc.z += v[q][r].z; acc.w += v[q][r].w; }
        // Peers may still be reading this CTA's partials: the sum goes to a
        // separate region holding this CTA's own rows.
        *reinterpret_cast<float4*>(cs + (p.n_tile + n / S) * CS_LD + m4) = acc;
      }
    }
  }
  cluster_sync();  // all remote reads done: no CTA's shared memory is needed by a peer any more
  {
    // Every warp stores. A thread writes 8 consecutive output columns (one
    // 16-byte vector) of one activation row per pass: 16 threads span a
    // 128-row tile, the CTA's threads NTHREADS / 16 rows n at a time. Rows
    // owned by this CTA: n = split + S j. What depends only on the thread's 8
    // columns is worked out once per tile, and two rows are loaded before
    // either is stored so that their shared-memory reads overlap.
    const float* cs = reinterpret_cast<const float*>(smem);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out[seg]);
    const int epi = p.epi[seg];
    const long long ldo = p.ldo[seg];
    constexpr int JSTEP = NTHREADS / 16;
    const int cg = threadIdx.x & 15, jr = threadIdx.x >> 4;
    const int n_own = (n_valid - split + S - 1) / S;
    const int half = p.d_r / 2;
    const float* rc = reinterpret_cast<const float*>(smem + p.rope_off);   // staged cos rows, then sin rows
    const int32_t* pos_s = reinterpret_cast<const int32_t*>(rc + p.n_tile * p.d_r);   // then positions, sequences
    for (int t = 0; t < MT; ++t) {
      const int mb = m0 + t * BM + cg * 8;  // first of this thread's 8 rows within the segment
      if (mb >= p.rows[seg]) continue;
      const int mcount = min(8, p.rows[seg] - mb);
      // the 8 columns' place in an output row, and whether and how they rotate
      long long col = 0;
      int j0 = 0, sg = 0;
      bool rope = false;
      if (epi == EPI_STORE) {
        col = z * p.bo[seg] + p.col0[seg] + mb;
      } else if (epi == EPI_SEGS) {
        // 8 rows inside one segment (seg_len % 8 == 0)
        const int sl = p.seg_len[seg];
        col = (long long)(mb / sl) * p.seg_stride[seg] + p.seg_off[seg] + mb % sl;
      } else if (epi == EPI_ROPE_SEGS) {
        // 8 rows of one rotated segment, all in one half of it (d_r % 16 == 0)
        sg = mb / p.d_r;
        j0 = mb % p.d_r;
        col = (long long)sg * p.seg_stride[seg] + p.seg_off[seg] + j0;
        rope = true;
      } else {  // EPI_APPEND: cache columns, the rotated ones past d_c
        col = p.col0[seg] + mb;
        if (col >= p.d_c) { j0 = (int)col - p.d_c; rope = true; }
      }
      const bool first = j0 < half;
      const int jj = first ? j0 : j0 - half;
      const int pcol = cg * 8 + (first ? half : -half);

      struct Row { float v[8]; __nv_bfloat16* dst; bool ok; };
      auto load = [&](int j, Row& r) {
        const int n = split + S * j;
        const float* row = S > 1 ? cs + (p.n_tile + j) * CS_LD : cs + (t * p.n_tile + n) * CS_LD;
        const long long gn = (long long)n0 + n;
        *reinterpret_cast<float4*>(r.v) = *reinterpret_cast<const float4*>(row + cg * 8);
        *reinterpret_cast<float4*>(r.v + 4) = *reinterpret_cast<const float4*>(row + cg * 8 + 4);
        r.ok = true;
        int ps = 0;
        if (epi == EPI_APPEND) {
          const int sq = p.rope_off ? pos_s[p.n_tile + n] : (p.tok_seq ? p.tok_seq[gn] : (int)gn);
          ps = p.rope_off ? pos_s[n] : p.tok_pos[gn];
          const bool seq_ok = sq >= 0 && sq < p.cache_batch;
          const bool pos_ok = ps >= 0 && ps < p.max_len && ps < p.max_pos;
          if (!seq_ok || !pos_ok) {
            if (col == 0) atomicOr(p.status, (seq_ok ? 0 : MLA_DEV_SEQ_RANGE) | (pos_ok ? 0 : MLA_DEV_POS_RANGE));
            r.ok = false;
            return;
          }
          r.dst = out + ((long long)sq * p.max_len + ps) * p.row_width + col;
        } else {
          r.dst = out + gn * ldo + col;
          if (rope) {
            ps = p.rope_off ? pos_s[n] : p.pos[gn];
            if (ps < 0 || ps >= p.max_pos) {
              if (j0 == 0 && sg == 0) atomicOr(p.status, MLA_DEV_QPOS_RANGE);
              ps = ps < 0 ? 0 : p.max_pos - 1;
            }
          }
        }
        if (rope) {
          const float* tc = p.rope_off ? rc + n * half + jj : p.rope_cos + (long long)ps * half + jj;
          const float* ts = p.rope_off ? rc + (p.n_tile + n) * half + jj : p.rope_sin + (long long)ps * half + jj;
          rope8(r.v, row + pcol, first, tc, ts);
        }
      };
      auto store = [&](const Row& r) {
        if (!r.ok) return;
        if (mcount == 8) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(r.v[2 * e], r.v[2 * e + 1]);
            pk[e] = *reinterpret_cast<uint32_t*>(&b2);
          }
          *reinterpret_cast<uint4*>(r.dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        } else {
          for (int e = 0; e < mcount; ++e) r.dst[e] = __float2bfloat16_rn(r.v[e]);
        }
      };
      int j = jr;
      for (; j + JSTEP < n_own; j += 2 * JSTEP) {
        Row a, b;
        load(j, a);
        load(j + JSTEP, b);
        store(a);
        store(b);
      }
      if (j < n_own) {
        Row a;
        load(j, a);
        store(a);
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

// The largest dynamic shared memory requested so far of one instantiation.
template <int CPB, bool TRANS>
cudaError_t ensure_smem(size_t smem_dyn) {
  static size_t smem_set = 0;
  if (smem_dyn <= smem_set) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<CPB, TRANS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_dyn);
  if (e == cudaSuccess) smem_set = smem_dyn;
  return e;
}

template <int CPB, bool TRANS>
cudaError_t launch_typed(const CUtensorMap* mw, const CUtensorMap& mx, const Params& p, dim3 grid, size_t smem_dyn,
                         cudaStream_t s) {  // mw: three weight maps
  cudaError_t e = ensure_smem<CPB, TRANS>(smem_dyn);
  if (e != cudaSuccess) return e;
  LaunchCfg lc(grid, dim3(NTHREADS), smem_dyn, s, (unsigned)p.splits);
  e = cudaLaunchKernelEx(&lc.cfg, gemm_tc_kernel<CPB, TRANS>, mw[0], mw[1], mw[2], mx, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int CPB, bool TRANS>
int max_clusters_typed(size_t smem_dyn, int S) {
  if (ensure_smem<CPB, TRANS>(smem_dyn) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute at{};
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = (unsigned)S;
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)S);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem_dyn;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<CPB, TRANS>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// How many clusters of S CTAs the device holds at once (the GPCs bound it:
// a cluster never spans two). Cached per configuration.
int max_clusters(int cpb, bool trans, size_t smem_dyn, int S) {
  struct Entry { int cpb, S; bool trans; size_t smem; int n; };
  static std::mutex mu;
  static std::vector<Entry> cache;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
      if (e.cpb == cpb && e.S == S && e.trans == trans && e.smem == smem_dyn) return e.n;
  }
  int n;
  if (trans) n = cpb == 4 ? max_clusters_typed<4, true>(smem_dyn, S) : cpb == 2 ? max_clusters_typed<2, true>(smem_dyn, S)
                                                                                : max_clusters_typed<1, true>(smem_dyn, S);
  else n = cpb == 4 ? max_clusters_typed<4, false>(smem_dyn, S) : cpb == 2 ? max_clusters_typed<2, false>(smem_dyn, S)
                                                                         : max_clusters_typed<1, false>(smem_dyn, S);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() < 256) cache.push_back(Entry{cpb, S, trans, smem_dyn, n});
  return n;
}

// One way to cut a launch into CTAs: CTAs per SM, 128-row tiles per CTA,
// K splits per tile, and the shared-memory layout that follows.
struct Choice {
  int per_sm, mt, S;
  int cpb, stage_bytes, kstages, nstage;
  int rope_off;   // where the epilogue's staged RoPE rows start (after the stages)
  size_t smem_dyn;
};

// Chunks per stage: as many as keep two stages within the budget (one stage
// if it is the only one), at most what the reduction has; the fp32 partial
// tiles [MT][n_tile][128] (plus the reduced own rows when split) reuse the
// stage buffers and must fit the budget too.
bool size_choice(Choice& c, int n_tile, int kchunks, int extra) {
  const int budget = (c.per_sm == 2 ? SMEM_TWO : SMEM_ONE) - extra;
  auto stage_of = [&](int cpb) { return c.mt * cpb * CHUNK_A + cpb * n_tile * 128; };
  int cpb = 4;
  while (cpb > 1 && (cpb > kchunks || 2 * stage_of(cpb) > budget) &&
         !(cpb <= kchunks && (kchunks + cpb - 1) / cpb == 1 && stage_of(cpb) <= budget))
    cpb >>= 1;
  c.cpb = cpb;
  c.stage_bytes = stage_of(cpb);
  if (c.stage_bytes > budget) return false;
  c.kstages = (kchunks + cpb - 1) / cpb;
  if (c.S > c.kstages) return false;
  c.nstage = budget / c.stage_bytes;
  if (c.nstage > 8) c.nstage = 8;
  if (c.nstage > c.kstages) c.nstage = c.kstages;
  const size_t cs = (size_t)c.mt * n_tile * CS_LD * 4 + (c.S > 1 ? (size_t)((n_tile + c.S - 1) / c.S) * CS_LD * 4 : 0);
  if (cs > (size_t)budget) return false;
  const size_t stages = (size_t)c.nstage * c.stage_bytes;
  c.rope_off = (int)(((cs > stages ? cs : stages) + 15) / 16 * 16);
  c.smem_dyn = (size_t)c.rope_off + extra + 1024;
  return true;
}

}  // namespace

bool gemm_tc_shape_ok(const TcGemm& g) {
  if (g.N <= 0 || g.K <= 0 || g.Z <= 0 || g.nseg < 1 || g.nseg > 3) return false;
  // Column chunks of 64 must not run past a row: the chunked views have no
  // per-row bound inside a chunk.
  if ((g.K % BK) || (g.ldx % 8) || (g.bx % 8) || (g.ldw % 8) || (g.bw % 8)) return false;
  if (reinterpret_cast<uintptr_t>(g.x) & 15) return false;
  if (g.nseg > 1 && g.w_transposed) return false;
  for (int s = 0; s < g.nseg; ++s) {
    if (g.rows[s] <= 0 || !g.w[s] || (reinterpret_cast<uintptr_t>(g.w[s]) & 15)) return false;
    if (g.w_transposed && (g.rows[s] % 64)) return false;
    // The epilogue stores 8 consecutive bf16 outputs (16 bytes) at a time;
    // RoPE keeps each group of 8 inside one half of a rotated segment, whose
    // partner rows share the 128-row tile.
    const int e = g.epi[s];
    if (!g.out[s] || (reinterpret_cast<uintptr_t>(g.out[s]) & 15)) return false;
    if ((g.ldo[s] % 8) || (g.bo[s] % 8) || (g.col0[s] % 8)) return false;
    if (e == EPI_ROPE_SEGS || e == EPI_APPEND) {
      if (g.d_r <= 0 || (BM % g.d_r) || (g.d_r % 16)) return false;
    }
    if ((e == EPI_ROPE_SEGS || e == EPI_SEGS) && ((g.seg_stride[s] % 8) || (g.seg_off[s] % 8))) return false;
    if (e == EPI_SEGS && (g.seg_len[s] <= 0 || (g.seg_len[s] % 8) || g.Z != 1)) return false;
    if (e == EPI_APPEND) {
      if ((g.row_width % 8) || (g.d_c % 8)) return false;
      // a cache segment is either inside the latent columns or exactly the rotated ones
      const bool latent = g.col0[s] + g.rows[s] <= g.d_c;
      const bool rope = g.col0[s] == g.d_c && g.rows[s] == g.d_r;
      if (!latent && !rope) return false;
    }
    if (e != EPI_STORE && e != EPI_ROPE_SEGS && e != EPI_APPEND && e != EPI_SEGS) return false;
  }
  return true;
}

cudaError_t launch_gemm_tc(const TcGemm& g, int num_sms, cudaStream_t s) {
  if (!gemm_tc_shape_ok(g)) return cudaErrorInvalidValue;
  Params p{};
  p.mstart[0] = 0;
  for (int sg = 0; sg < 3; ++sg) {
    const bool on = sg < g.nseg;
    p.rows[sg] = on ? g.rows[sg] : 0;
    p.col0[sg] = on ? g.col0[sg] : 0;
    p.epi[sg] = on ? g.epi[sg] : EPI_STORE;
    p.out[sg] = on ? g.out[sg] : nullptr;
    p.ldo[sg] = on ? g.ldo[sg] : 0;
    p.bo[sg] = on ? g.bo[sg] : 0;
    p.seg_stride[sg] = on ? g.seg_stride[sg] : 0;
    p.seg_off[sg] = on ? g.seg_off[sg] : 0;
    p.seg_len[sg] = on ? g.seg_len[sg] : 0;
    p.mstart[sg + 1] = p.mstart[sg] + (on ? (g.rows[sg] + BM - 1) / BM : 0);
  }
  p.mtiles_total = p.mstart[3];
  p.N = g.N; p.K = g.K; p.Z = g.Z;
  // Activation tiles of up to 256 rows for decode-sized batches (one tile);
  // with more tokens, tiles of 128 rows, whose fp32 partial tile leaves room
  // for two CTAs per SM (one's epilogue runs beside the other's stream):
  // measured 4-12 % faster on the MHA path's projections (8192 tokens).
  p.n_tile = g.N > 256 ? 128 : (g.N >= 256 ? 256 : ((g.N + 15) / 16) * 16);
  const int kchunks = g.K / BK;
  const long long n_tiles = (g.N + p.n_tile - 1) / p.n_tile;
  if (n_tiles > 65535 || g.Z > 65535) return cudaErrorInvalidValue;
  if (num_sms < 1) num_sms = 1;
  const long long tiles_all = (long long)p.mtiles_total * n_tiles * g.Z;
  bool mt_ok = true;
  for (int sg = 0; sg < g.nseg; ++sg) mt_ok = mt_ok && g.epi[sg] != EPI_APPEND;
  auto mt_fits = [&](int c) {
    return mt_ok && p.mtiles_total % c == 0 && p.mstart[1] % c == 0 && p.mstart[2] % c == 0 && c * p.n_tile <= 512;
  };
  Choice best{};
  bool have = false;
  // With one activation tile (decode) a RoPE or cache-row epilogue stages
  // its per-row positions and cos/sin rows in shared memory (stage_rope).
  bool roped = false;
  for (int sg = 0; sg < g.nseg; ++sg) roped = roped || g.epi[sg] == EPI_ROPE_SEGS || g.epi[sg] == EPI_APPEND;
  const int rope_extra = roped ? p.n_tile * (g.d_r * 4 + 8) : 0;
  if (n_tiles == 1) {
    // Decode-sized N (one activation tile): the launch is one wave, and its
    // time is the larger of the weights' HBM time and the busiest SM's copy
    // time (an SM lands about 85 GB/s of TMA boxes). Among the ways to cut it
    // (CTAs per SM, tiles per CTA sharing their activations, K splits over a
    // cluster that the GPCs can hold at once) take the fastest estimate; a
    // split costs its cluster sum. The estimate leaves out the epilogue, which
    // is latency-bound and shorter with fewer tiles per CTA and more CTAs per
    // SM, so estimates within 15 % count as a tie and go to more CTAs.
    const double hbm_s = ((double)p.mtiles_total * BM * g.K + (double)g.N * g.K) * 2.0 * g.Z / 6.3e12;
    double best_t = 0;
    long long best_ctas = 0;
    for (int per_sm = 1; per_sm <= 2; ++per_sm)
      for (int mt = 1; mt <= MAX_MT; mt *= 2)
        for (int S = 1; S <= MAX_SPLITS; ++S) {
          if (mt > 1 && (S > 1 || !mt_fits(mt))) continue;
          Choice c{per_sm, mt, S};
          if (!size_choice(c, p.n_tile, kchunks, rope_extra)) continue;
          const long long groups = tiles_all / mt, ctas = groups * S;
          if (ctas > (long long)per_sm * num_sms) continue;
          if (S > 1 && groups > max_clusters(c.cpb, g.w_transposed != 0, c.smem_dyn, S)) continue;
          const double cta_bytes = (double)((c.kstages + S - 1) / S) * c.stage_bytes;
          const double busiest = (double)((ctas + num_sms - 1) / num_sms) * cta_bytes;
          const double t = (hbm_s > busiest / 85e9 ? hbm_s : busiest / 85e9) + (S > 1 ? 1e-6 : 0.0);
          const bool better = ctas > best_ctas ? t <= best_t * 1.15 : t * 1.15 < best_t;
          if (!have || better) {
            best = c;
            best_t = t;
            best_ctas = ctas;
            have = true;
          }
        }
  }
  if (!have) {
    // Many activation tiles (several tokens per sequence): when the tiles
    // outnumber the SMs two CTAs share an SM (half the stage budget each,
    // when the fp32 partial tile fits it) so that every tile is resident at
    // once, and a CTA takes several tiles sharing their activations; else
    // one CTA per SM keeps the most bytes in flight per tile and the
    // reduction is split over a cluster.
    Choice c{};
    c.per_sm = (tiles_all > num_sms && (size_t)p.n_tile * CS_LD * 4 <= (size_t)SMEM_TWO) ? 2 : 1;
    const int slots = num_sms * c.per_sm;
    const int budget = c.per_sm == 2 ? SMEM_TWO : SMEM_ONE;
    c.mt = 1;
    if (tiles_all > slots)
      for (int m = 2; m <= MAX_MT; m *= 2)
        if (mt_fits(m) && (size_t)m * p.n_tile * CS_LD * 4 <= (size_t)budget) {
          c.mt = m;
          if (tiles_all / m <= slots) break;
        }
    const long long tiles = tiles_all / c.mt;
    long long S = tiles >= slots ? 1 : slots / tiles;
    if (S > MAX_SPLITS) S = MAX_SPLITS;
    if (c.mt > 1 || S < 1) S = 1;
    c.S = (int)S;
    while (!size_choice(c, p.n_tile, kchunks, 0)) {
      if (c.S > 1) { --c.S; continue; }
      return cudaErrorInvalidValue;
    }
    best = c;
  }
  const int mt = best.mt, cpb = best.cpb;
  p.mt = mt;
  p.splits = best.S;
  p.stage_bytes = best.stage_bytes;
  p.kstages = best.kstages;
  p.nstage = best.nstage;
  const size_t smem_dyn = best.smem_dyn;
  const long long S = best.S;
  p.rope_off = have && roped ? best.rope_off : 0;
  p.tmem_cols = pow2_at_least((uint32_t)(mt * p.n_tile));
  p.idesc = idesc_bf16(BM, p.n_tile, g.w_transposed != 0, false);
  p.rope_cos = g.rope_cos; p.rope_sin = g.rope_sin; p.d_r = g.d_r; p.max_pos = g.max_pos;
  p.pos = g.pos;
  p.tok_seq = g.tok_seq; p.tok_pos = g.tok_pos; p.cache_batch = g.cache_batch; p.max_len = g.max_len;
  p.d_c = g.d_c; p.row_width = g.row_width; p.status = g.status;

  // Tensor maps, all 4-D with the column chunk outside the row:
  //   weights    {64, rows, K/64, Z}   box {64, 128, CPB, 1}
  //   transposed {64, K, rows/64, Z}   box {64, 64 CPB, 2, 1}   (stored [K][rows])
  //   activation {64, N, K/64, Z}      box {64, n_tile, CPB, 1}
  CUtensorMap mw[3], mx;
  for (int sg = 0; sg < 3; ++sg) {
    const int src = sg < g.nseg ? sg : 0;
    uint64_t dims[4], strides[3];
    uint32_t box[4];
    // with one batch the outer stride is never stepped; give it the tensor's size
    const uint64_t zstride = g.Z > 1 ? (uint64_t)g.bw * 2
                                     : (uint64_t)(g.w_transposed ? g.K : g.rows[src]) * (uint64_t)g.ldw * 2;
    if (g.w_transposed) {
      dims[0] = 64; dims[1] = (uint64_t)g.K; dims[2] = (uint64_t)g.rows[src] / 64; dims[3] = (uint64_t)g.Z;
      strides[0] = (uint64_t)g.ldw * 2; strides[1] = 128; strides[2] = zstride;
      box[0] = 64; box[1] = (uint32_t)(cpb * BK); box[2] = 2; box[3] = 1;
    } else {
      dims[0] = 64; dims[1] = (uint64_t)g.rows[src]; dims[2] = (uint64_t)kchunks; dims[3] = (uint64_t)g.Z;
      strides[0] = (uint64_t)g.ldw * 2; strides[1] = 128; strides[2] = zstride;
      box[0] = 64; box[1] = BM; box[2] = (uint32_t)cpb; box[3] = 1;
    }
    if (!make_tmap_4d_bf16_sw128(&mw[sg], g.w[src], dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    uint64_t dims[4] = {64, (uint64_t)g.N, (uint64_t)kchunks, (uint64_t)g.Z};
    uint64_t strides[3] = {(uint64_t)g.ldx * 2, 128, g.Z > 1 ? (uint64_t)g.bx * 2 : (uint64_t)g.N * g.ldx * 2};
    uint32_t box[4] = {64, (uint32_t)p.n_tile, (uint32_t)cpb, 1};
    if (!make_tmap_4d_bf16_sw128(&mx, g.x, dims, strides, box)) return cudaErrorInvalidValue;
  }

  const dim3 grid((unsigned)(p.mtiles_total / mt * S), (unsigned)n_tiles, (unsigned)g.Z);
  if (g.w_transposed) {
    if (cpb == 4) return launch_typed<4, true>(mw, mx, p, grid, smem_dyn, s);
    if (cpb == 2) return launch_typed<2, true>(mw, mx, p, grid, smem_dyn, s);
    return launch_typed<1, true>(mw, mx, p, grid, smem_dyn, s);
  }
  if (cpb == 4) return launch_typed<4, false>(mw, mx, p, grid, smem_dyn, s);
  if (cpb == 2) return launch_typed<2, false>(mw, mx, p, grid, smem_dyn, s);
  return launch_typed<1, false>(mw, mx, p, grid, smem_dyn, s);
}

}  // namespace mla
