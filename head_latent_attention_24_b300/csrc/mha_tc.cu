// Tensor-core causal multi-head attention over materialised keys and values,
// for the DeepSeek-V2 head shape (d_h = 128, d_r = 64, bf16): the MHA path of
// several new tokens per sequence (page "Latent 压缩": at prefill MLA takes the
// MHA path; page "MiniMind 学习笔记 10", §10 naive version, §12 causal
// visibility with a cache; page "MLA：潜在表示压缩与解耦 RoPE", §6 k = [k_C ; k_R]
// with the RoPE key shared by the heads, §7 scale 1/sqrt(d_h + d_r)).
//
// One CTA per (128 queries, head, sequence). The query tile (128 x 192) is
// moved into TMEM once and is the A operand of every QK; key tiles of 128 rows
// stream through two TMA rings, a two-stage one for k_C (128 x 128) with the
// shared k_R (128 x 64, read straight from the cache rows), freed after the
// tile's QK, and a three-stage one for v_C (128 x 128), freed after its PV.
// Per key tile:
//   S = Q . K^T      M = 128 queries, N = 128 keys, K = 192   (TMEM)
//   P = 2^(S*scale*log2e - m)  in bf16, written by the softmax threads into TMEM
//   O += P . V       M = 128 queries, N = 128 (d_h), K = 128 keys, A from TMEM
// Each query row (a TMEM lane) belongs to two softmax threads, one per half of
// the key tile; they exchange the row's tile maximum, the reference maximum
// moves lazily (only when a tile's maximum rises
// more than 8 above it, when the thread rescales its row of O in TMEM), and
// rows a query may not see (later positions) get P = 0; v_C rows past the last
// query's position are zeroed in shared memory before PV reads them. The QK of
// tile j+1 runs on the tensor core while the softmax works on tile j.
//
// Warp 0 issues TMA, warp 1 owns TMEM and issues the QK MMAs, warp 2 the PV
// MMAs, warps 3-10 run the softmax and the epilogue (two warps per query row,
// each with half of the tile's keys). Every mbarrier wait is bounded;
// on expiry the CTA records MLA_DEV_TIMEOUT, stops issuing work, waits
// (bounded) for its own copies in flight and frees its TMEM.
#include "internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int DH = 128, DR = 64, DQ = DH + DR;   // the head shape this kernel serves
constexpr int TQ = 128;                           // queries per CTA (MMA M)
constexpr int TK = 128;                           // keys per tile (MMA N of QK, K of PV)
constexpr int NTHREADS = 352;
constexpr long long WAIT_CYCLES = 4000000000LL;   // ~2 s
constexpr float kLn2 = 0.693147180559945309f;
constexpr float RESCALE_THRESHOLD = 8.0f;

constexpr int CHUNK = TK * 128;                   // 16 KB: 128 rows x 64 bf16 (128 B, swizzled)
// Keys and values in rings of their own: a key stage (k_C, 2 chunks, and k_R,
// 1 chunk) is free once its QK has run, a value stage (v_C, 2 chunks) once its
// PV has; the next loads of each start that early. The value ring is the
// deeper one: a value load is issued only when the PV two (three) tiles back
// has run, and the PV it feeds comes right after the softmax.
constexpr int KSTAGE = 3 * CHUNK, VSTAGE = 2 * CHUNK;
constexpr int NKS = 2, NVS = 3;
constexpr int KRING_OFF = 0;
constexpr int VRING_OFF = KRING_OFF + NKS * KSTAGE;
constexpr int SMEM_DYN = VRING_OFF + NVS * VSTAGE + 1024;
// The query tile lands in key stage 1 (3 chunks, the size of a key stage);
// the softmax warps move it into TMEM, where it is the A operand of QK, and
// hand the stage back for key tile 1.
constexpr int Q_STAGE = 1;
// TMEM columns
constexpr uint32_t S_COL = 0;                     // 128 fp32
constexpr uint32_t O_COL = 128;                   // 128 fp32
constexpr uint32_t P_COL = 256;                   // 64: 128 bf16 packed two per column
constexpr uint32_t Q_COL = 320;                   // 96: 192 bf16 packed two per column
constexpr uint32_t TMEM_COLS = 512;

struct Ctl {
  uint64_t q_full, q_ready, k_full[NKS], k_empty[NKS], v_full[NVS], v_empty[NVS];
  uint64_t s_full, s_free, p_full, pv_done, mma_done;
  uint32_t tmem_base;
  int abort;
  long long wait_limit;
  float mx[2][2][TQ];   // per tile parity, key half and query row: the half's tile maximum
  float ls[2][TQ];      // per key half and query row: the half's softmax sum
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Ctl& ctl, int32_t* status) {
  volatile int* ab = reinterpret_cast<volatile int*>(&ctl.abort);
  if (*ab) return false;
  if (mbar_wait_abortable(bar, parity, ctl.wait_limit, ab)) return true;
  if (!*ab) atomicOr(status, MLA_DEV_TIMEOUT);
  *ab = 1;
  return false;
}

__device__ __forceinline__ void drain_ring(uint64_t* full, int ring, int issued) {
  for (int s = 0; s < ring; ++s) {
    if (issued <= s) break;
    const int last = s + ring * ((issued - 1 - s) / ring);
    mbar_wait(&full[s], (uint32_t)((last / ring) & 1), WAIT_CYCLES / 8);
  }
}

// The two softmax warps of TMEM lane quarter q (named barrier 1 + q, 64 threads).
__device__ __forceinline__ void pair_sync(int quarter) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory");
}
__device__ __forceinline__ bool pair_all(int quarter, bool v) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n barrier.cta.red.and.pred po, %2, 64, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(1 + quarter)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(NTHREADS, 1)
    mha_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_kr,
                  const MhaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Ctl ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * TQ, head = blockIdx.y, b = blockIdx.z;

  if (threadIdx.x == 0) {
    mbar_init(&ctl.q_full, 1);
    mbar_init(&ctl.q_ready, 8);
    for (int i = 0; i < NKS; ++i) { mbar_init(&ctl.k_full[i], 1); mbar_init(&ctl.k_empty[i], 1); }
    for (int i = 0; i < NVS; ++i) { mbar_init(&ctl.v_full[i], 1); mbar_init(&ctl.v_empty[i], 1); }
    mbar_init(&ctl.s_full, 1);
    mbar_init(&ctl.s_free, 8);
    mbar_init(&ctl.p_full, 8);
    mbar_init(&ctl.pv_done, 1);
    mbar_init(&ctl.mma_done, 2);
    ctl.abort = 0;
    ctl.wait_limit = a.wait_cycles > 0 ? a.wait_cycles : WAIT_CYCLES;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl.tmem_base;
  pdl_trigger();
  pdl_wait();   // q, k_c and v_c come from earlier kernels

  // The queries of this tile sit at positions qp0 .. qp0 + nq - 1 and see keys
  // 0 .. qp_last; key tiles 0 .. nk - 1 cover them.
  int pos0 = a.q_pos0[b];
  if (pos0 < 0 || pos0 > a.max_len - a.T) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && head == 0) atomicOr(a.status, MLA_DEV_QPOS_RANGE);
    pos0 = pos0 < 0 ? 0 : a.max_len - a.T;
  }
  const int nq = min(TQ, a.T - q0);
  const int qp0 = pos0 + q0, qp_last = qp0 + nq - 1;
  const int nk = qp_last / TK + 1;
  const uint32_t sbase = smem_u32(smem);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producers
    // lane 0: the queries, then the key stages; lane 1: the value stages
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_kr);
      const int qrow = b * a.T + q0;
      mbar_arrive_expect_tx(&ctl.q_full, 3 * CHUNK);
      tma_load_3d(smem + KRING_OFF + Q_STAGE * KSTAGE, &map_q, &ctl.q_full, 0, qrow, head * 3);
      int i = 0;
      bool ok = true;
      for (; i < nk; ++i) {
        const int st = i % NKS;
        if (i >= NKS) ok = wait_or_abort(&ctl.k_empty[st], ((i / NKS) - 1) & 1, ctl, a.status);
        else if (st == Q_STAGE) ok = wait_or_abort(&ctl.q_ready, 0, ctl, a.status);   // the queries have left
        if (!ok) break;
        uint8_t* dst = smem + KRING_OFF + st * KSTAGE;
        const int krow = b * a.max_len + i * TK;
        mbar_arrive_expect_tx(&ctl.k_full[st], KSTAGE);
        tma_load_3d(dst, &map_k, &ctl.k_full[st], 0, krow, head * 2);
        tma_load_2d(dst + 2 * CHUNK, &map_kr, &ctl.k_full[st], 0, krow);
      }
      if (!ok) {   // no copy lands after the CTA moves on
        drain_ring(ctl.k_full, NKS, i);
        mbar_wait(&ctl.q_full, 0, WAIT_CYCLES / 8);
      }
    } else if (lane == 1) {
      prefetch_tensormap(&map_v);
      int i = 0;
      bool ok = true;
      for (; i < nk; ++i) {
        const int st = i % NVS;
        if (i >= NVS) ok = wait_or_abort(&ctl.v_empty[st], ((i / NVS) - 1) & 1, ctl, a.status);
        if (!ok) break;
        mbar_arrive_expect_tx(&ctl.v_full[st], VSTAGE);
        tma_load_3d(smem + VRING_OFF + st * VSTAGE, &map_v, &ctl.v_full[st], 0, b * a.max_len + i * TK, head * 2);
      }
      if (!ok) drain_ring(ctl.v_full, NVS, i);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK issuer
    // S(j) = Q . K(j)^T (Q from TMEM) once key stage j has landed and the
    // softmax has read S(j-1). QK and PV have an issuing thread each, so that
    // a PV never waits behind the next tile's load.
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16(TQ, TK, false, false);
      const uint64_t k_desc = sdesc_sw128(sbase + KRING_OFF, 16, 1024);
      bool ok = wait_or_abort(&ctl.q_ready, 0, ctl, a.status);
      for (int j = 0; j < nk && ok; ++j) {
        const int st = j % NKS;
        ok = wait_or_abort(&ctl.k_full[st], (j / NKS) & 1, ctl, a.status) &&
             (j < 1 || wait_or_abort(&ctl.s_free, (j - 1) & 1, ctl, a.status));
        if (!ok) break;
        tc_fence_after();
        const uint64_t kd = k_desc + (uint64_t)((st * KSTAGE) >> 4);
#pragma unroll
        for (int c = 0; c < 3; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_ta(tbase + S_COL, tbase + Q_COL + c * 32 + k * 8, kd + (uint64_t)((c * CHUNK + k * 32) >> 4),
                        IDESC_QK, (c > 0 || k > 0) ? 1u : 0u);
        mma_commit(&ctl.s_full);
        mma_commit(&ctl.k_empty[st]);   // the key stage: its QK is done
      }
      // nothing of this CTA's reaches the tensor cores after it moves on
      mma_commit(&ctl.mma_done);
      mbar_wait(&ctl.mma_done, 0, WAIT_CYCLES / 8);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ PV issuer
    // O += P(j) . V(j) once the softmax has written P(j) and V(j) has landed;
    // the value stage is free when this PV completes.
    if (lane == 0) {
      constexpr uint32_t IDESC_PV = idesc_bf16(TQ, DH, false, true);
      const uint64_t v_desc = sdesc_sw128(sbase + VRING_OFF, CHUNK, 1024);
      bool ok = true;
      for (int j = 0; j < nk && ok; ++j) {
        const int st = j % NVS;
        ok = wait_or_abort(&ctl.p_full, j & 1, ctl, a.status) &&
             wait_or_abort(&ctl.v_full[st], (j / NVS) & 1, ctl, a.status);
        if (!ok) break;
        tc_fence_after();
        const uint64_t vd = v_desc + (uint64_t)((st * VSTAGE) >> 4);
#pragma unroll
        for (int k = 0; k < TK / 16; ++k)
          mma_bf16_ta(tbase + O_COL, tbase + P_COL + k * 8, vd + (uint64_t)((k * 2048) >> 4), IDESC_PV,
                      (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(&ctl.pv_done);
        mma_commit(&ctl.v_empty[st]);
      }
      mma_commit(&ctl.mma_done);
      mbar_wait(&ctl.mma_done, 0, WAIT_CYCLES / 8);
    }
  } else {
    // ------------------------------------------------------------ softmax warps 3..10
    // Two warps per TMEM lane quarter: warps 3..6 and 7..10 share query rows
    // 32q..32q+31 (one row per lane), each taking 64 of the tile's keys and 64
    // of O's columns; they meet (named barrier 1+q, 64 threads) to agree on
    // every wait's outcome and to exchange row maxima and sums.
    const int quarter = warp & 3, half = (warp - 3) >> 2;
    const int r = quarter * 32 + lane;                 // TMEM lane = query row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int qp = qp0 + r;                            // this row's position (rows past nq: not stored)
    const float sl2 = a.scale_log2;
    constexpr int HK = TK / 2;                         // keys per half
    float m_ref = -INFINITY, l = 0.f;
    // The query tile from key stage Q_STAGE into TMEM (row r = lane r, 32
    // columns per 64-column chunk): half 0 moves chunks 0 and 1, half 1 chunk 2.
    bool ok = pair_all(quarter, __all_sync(0xffffffffu, wait_or_abort(&ctl.q_full, 0, ctl, a.status)));
    if (ok) {
      const uint8_t* qs = smem + KRING_OFF + Q_STAGE * KSTAGE + (r >> 3) * 1024 + (r & 7) * 128;
      for (int c = half * 2; c < (half == 0 ? 2 : 3); ++c) {
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = *reinterpret_cast<const uint4*>(qs + c * CHUNK + ((v ^ (r & 7)) << 4));
          w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
        }
        tmem_st32(tbase + lane_base + Q_COL + c * 32, w);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.q_ready);   // also: the stage may take key tile 1
    }
    for (int j = 0; j < nk && ok; ++j) {
      const int k0 = j * TK + half * HK;
      ok = pair_all(quarter, __all_sync(0xffffffffu, wait_or_abort(&ctl.s_full, j & 1, ctl, a.status)));
      if (!ok) break;
      tc_fence_after();
      float s[HK];
      tmem_ld32(tbase + lane_base + S_COL + half * HK, s);
      tmem_ld32(tbase + lane_base + S_COL + half * HK + 32, s + 32);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.s_free);
      // causal mask: key k0 + c is visible to this row when k0 + c <= qp
      const int nvis = max(0, min(HK, qp - k0 + 1));
      // Tiles below the diagonal (every key visible to every row of the warp)
      // take the short path: the maximum of the raw scores, scaled once, and
      // the scale folded into the exponent's FMA.
      const bool full = __all_sync(0xffffffffu, nvis == HK);
      float mx = -INFINITY;
      if (full) {
#pragma unroll
        for (int c = 0; c < HK; ++c) mx = fmaxf(mx, s[c]);
        mx *= sl2;
      } else {
#pragma unroll
        for (int c = 0; c < HK; ++c) {
          s[c] = c < nvis ? s[c] * sl2 : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
      }
      ctl.mx[j & 1][half][r] = mx;
      pair_sync(quarter);
      mx = fmaxf(mx, ctl.mx[j & 1][half ^ 1][r]);   // the row's tile maximum, the same in both halves
      float alpha = 1.f;
      if (mx > m_ref + RESCALE_THRESHOLD) {   // also the first tile a row sees anything (m_ref = -inf)
        alpha = ex2_approx(m_ref - mx);
        m_ref = mx;
      }
      uint32_t pk[HK / 2];
      float lsum0 = 0.f, lsum1 = 0.f;   // the softmax sum from the unrounded weights
      if (full) {
        const float neg = -m_ref;
#pragma unroll
        for (int c = 0; c < HK; c += 2) {
          const float p0 = ex2_approx(fmaf(s[c], sl2, neg)), p1 = ex2_approx(fmaf(s[c + 1], sl2, neg));
          lsum0 += p0;
          lsum1 += p1;
          pk[c / 2] = pack_bf16(p0, p1);
        }
      } else {
#pragma unroll
        for (int c = 0; c < HK; c += 2) {
          const float p0 = c < nvis ? ex2_approx(s[c] - m_ref) : 0.f;
          const float p1 = c + 1 < nvis ? ex2_approx(s[c + 1] - m_ref) : 0.f;
          lsum0 += p0;
          lsum1 += p1;
          pk[c / 2] = pack_bf16(p0, p1);
        }
      }
      l = l * alpha + (lsum0 + lsum1);   // this half's share of the row sum
      // P(j) replaces P(j-1) in TMEM and O is rescaled: both only after PV(j-1)
      if (j > 0) {
        ok = pair_all(quarter, __all_sync(0xffffffffu, wait_or_abort(&ctl.pv_done, (j - 1) & 1, ctl, a.status)));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < DH / 2; c += 32) {
            float v[32];
            tmem_ld32(tbase + lane_base + O_COL + half * (DH / 2) + c, v);
            tmem_ld_wait();
            uint32_t w[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(v[e] * alpha);
            tmem_st32(tbase + lane_base + O_COL + half * (DH / 2) + c, w);
          }
        }
      }
      tmem_st32(tbase + lane_base + P_COL + half * (HK / 2), pk);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      // the last tile's v_C rows past the last query's position may hold
      // anything (rows no query of this tile may see): zero them in the stage
      // before PV reads it (each warp a share of the rows; its p_full arrival
      // below publishes them)
      if (j == nk - 1 && qp_last - j * TK + 1 < TK) {
        const int st = j % NVS;
        ok = pair_all(quarter, __all_sync(0xffffffffu, wait_or_abort(&ctl.v_full[st], (j / NVS) & 1, ctl, a.status)));
        if (!ok) break;
        const int first = qp_last - j * TK + 1;   // rows first .. TK-1 of both v_C chunks
        uint8_t* vbase = smem + VRING_OFF + st * VSTAGE;
        const int tid = threadIdx.x - 96;
        for (int w = tid; w < (TK - first) * 16; w += 256) {
          const int row = first + w / 16, part = w % 16;   // 8 x 16 B per row and chunk
          *reinterpret_cast<uint4*>(vbase + (part >> 3) * CHUNK + row * 128 + (part & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.p_full);
    }
    // ---------------------------------------------------------------- epilogue
    if (ok) ok = pair_all(quarter, __all_sync(0xffffffffu, wait_or_abort(&ctl.pv_done, (nk - 1) & 1, ctl, a.status)));
    if (ok) {
      ctl.ls[half][r] = l;
      pair_sync(quarter);
      l += ctl.ls[half ^ 1][r];
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool store = r < nq;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) + (((size_t)b * a.T + q0 + r) * a.n_h + head) * DH;
#pragma unroll 1
      for (int c = half * (DH / 2); c < (half + 1) * (DH / 2); c += 32) {
        float v[32];
        tmem_ld32(tbase + lane_base + O_COL + c, v);
        tmem_ld_wait();
        if (store) {
#pragma unroll
          for (int e = 0; e < 32; e += 8)
            *reinterpret_cast<uint4*>(orow + c + e) =
                make_uint4(pack_bf16(v[e] * inv_l, v[e + 1] * inv_l), pack_bf16(v[e + 2] * inv_l, v[e + 3] * inv_l),
                           pack_bf16(v[e + 4] * inv_l, v[e + 5] * inv_l), pack_bf16(v[e + 6] * inv_l, v[e + 7] * inv_l));
        }
      }
      if (store && half == 0) a.lse[((size_t)b * a.T + q0 + r) * a.n_h + head] = (m_ref + log2f(l)) * kLn2;
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, TMEM_COLS);
}

}  // namespace

bool mha_tc_supported(const mla_handle_s* h) {
  const mla_config_t& c = h->cfg;
  return c.dtype == MLA_BF16 && c.d_h == DH && c.d_r == DR && c.d_c % 8 == 0;
}

cudaError_t launch_mha_tc(const MhaArgs& a, cudaStream_t s) {
  if (a.d_h != DH || a.d_r != DR || a.T <= 0 || a.B <= 0 || a.n_h <= 0) return cudaErrorInvalidValue;
  if (a.n_h > 65535 || a.B > 65535) return cudaErrorInvalidValue;
  const int D = a.d_c + a.d_r;
  CUtensorMap map_q, map_k, map_v, map_kr;
  // q [B*T rows][n_h * 192] and k_c / v_c [B*max_len rows][n_h * 128] through
  // 3-D views {64 columns, rows, 64-column chunks} (chunk outermost), so one
  // box brings a head's 3 (q) or 2 (k_c, v_c) chunks of 128 rows chunk-major:
  // one TMA operation each, the operation count (not the bytes) being what
  // limits an SM's copy rate for 16 KB boxes. The cache's RoPE columns
  // [B*max_len rows][64] from column d_c: one 64 x 128-row box.
  {
    const uint64_t dq[3] = {64, (uint64_t)a.B * a.T, (uint64_t)a.n_h * 3};
    const uint64_t sq[2] = {(uint64_t)a.n_h * DQ * 2, 128};
    const uint32_t bq[3] = {64, TQ, 3};
    if (!make_tmap_3d_bf16_sw128(&map_q, a.q, dq, sq, bq)) return cudaErrorInvalidValue;
    const uint64_t dk[3] = {64, (uint64_t)a.B * a.max_len, (uint64_t)a.n_h * 2};
    const uint64_t sk[2] = {(uint64_t)a.n_h * DH * 2, 128};
    const uint32_t bk[3] = {64, TK, 2};
    if (!make_tmap_3d_bf16_sw128(&map_k, a.k_c, dk, sk, bk)) return cudaErrorInvalidValue;
    if (!make_tmap_3d_bf16_sw128(&map_v, a.v_c, dk, sk, bk)) return cudaErrorInvalidValue;
  }
  const char* rope = static_cast<const char*>(a.cache) + (size_t)a.d_c * 2;
  if (!make_tmap_2d_bf16(&map_kr, rope, DR, (uint64_t)a.B * a.max_len, (uint64_t)D * 2, 64, TK, 128))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(mha_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  LaunchCfg lc(dim3((unsigned)((a.T + TQ - 1) / TQ), (unsigned)a.n_h, (unsigned)a.B), dim3(NTHREADS), SMEM_DYN, s);
  cudaError_t e = cudaLaunchKernelEx(&lc.cfg, mha_tc_kernel, map_q, map_k, map_v, map_kr, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
