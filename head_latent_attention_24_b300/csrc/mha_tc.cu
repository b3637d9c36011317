// Tensor-core causal multi-head attention over materialised keys and values,
// for the DeepSeek-V2 head shape (d_h = 128, d_r = 64, bf16): the MHA path of
// several new tokens per sequence (page "Latent 压缩": at prefill MLA takes the
// MHA path; page "MiniMind 学习笔记 10", §10 naive version, §12 causal
// visibility with a cache; page "MLA：潜在表示压缩与解耦 RoPE", §6 k = [k_C ; k_R]
// with the RoPE key shared by the heads, §7 scale 1/sqrt(d_h + d_r)).
//
// One CTA per SM runs work items of 128 queries of one head of one sequence,
// taken at run time (Item, item_of below). An item's query tile (128 x 192)
// is moved into TMEM and is the A operand of every QK; key tiles of 128 rows
// stream through two TMA rings, a two-stage one for k_C (128 x 128) with the
// shared k_R (128 x 64, read straight from the cache rows), freed after the
// tile's QK, and a three-stage one for v_C (128 x 128), freed after its PV. The next
// item's query tile comes through the key ring behind the current item's
// keys and goes into TMEM as soon as the current item's last scores are read,
// so its first QK runs during the current item's last PV and epilogue.
// Per key tile:
//   S = Q . K^T      M = 128 queries, N = 128 keys, K = 192   (TMEM)
//   P = 2^(S*scale*log2e - m)  in bf16, written by the softmax threads into TMEM
//   O += P . V       M = 128 queries, N = 128 (d_h), K = 128 keys, A from TMEM
// Each query row (a TMEM lane) belongs to two softmax threads, one per half of
// the key tile; they exchange the row's tile maximum, the reference maximum
// moves lazily (only when a tile's maximum rises more than 8 above it, when
// the thread rescales its row of O in TMEM), and
// rows a query may not see (later positions) get P = 0; v_C rows past the last
// query's position are zeroed in shared memory before PV reads them. The QK of
// tile j+1 runs on the tensor core while the softmax works on tile j.
//
// Warp 0 issues TMA, warp 1 owns TMEM and issues the QK MMAs, warp 2 the PV
// MMAs, warps 3-10 move the queries and run the softmax and the epilogue (two
// warps per query row, each with half of the tile's keys). Every mbarrier
// wait is bounded; on expiry the CTA records MLA_DEV_TIMEOUT, stops issuing
// work, waits (bounded) for its own copies in flight and frees its TMEM.
#include <atomic>

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
// TMEM columns
constexpr uint32_t S_COL = 0;                     // 128 fp32
constexpr uint32_t O_COL = 128;                   // 128 fp32
constexpr uint32_t P_COL = 256;                   // 64: 128 bf16 packed two per column
constexpr uint32_t Q_COL = 320;                   // 96: 192 bf16 packed two per column
constexpr uint32_t TMEM_COLS = 512;

// Work items are handed out at run time: the key-ring producer takes the next
// item index from a per-launch device counter and passes it to the other
// roles through a small ring in shared memory (NIR entries; the readers are
// the value producer, both MMA issuers and the eight softmax warps).
constexpr int NIR = 4, IR_READERS = 11;
constexpr int NCTR = 64;   // launches in flight that may use the counters at once
__device__ unsigned int g_item_next[NCTR];
__device__ unsigned int g_cta_done[NCTR];

struct Ctl {
  uint64_t q_ready, k_full[NKS], k_empty[NKS], v_full[NVS], v_empty[NVS];
  uint64_t ir_full[NIR], ir_empty[NIR];
  int ir_item[NIR];
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

// One work item: 128 queries of one head of one sequence. Items are numbered
// sequence- and head-major and, inside a head, longest key range first (the
// last query tile first): the CTAs working at one time share a few heads'
// keys and values in L2, and the short items come last.
struct Item {
  int q0, head, b;   // first query of the tile, head, sequence
  int qp0, nq, nk;   // position of the first query, queries in the tile, key tiles
  int qp_last;
};

__device__ __forceinline__ Item item_of(const MhaArgs& a, int k, bool flag) {
  const int nqt = (a.T + TQ - 1) / TQ;
  Item it;
  const int bh = k / nqt, qt = nqt - 1 - k % nqt;
  it.b = bh / a.n_h;
  it.head = bh % a.n_h;
  it.q0 = qt * TQ;
  int pos0 = a.q_pos0[it.b];
  if (pos0 < 0 || pos0 > a.max_len - a.T) {
    if (flag) atomicOr(a.status, MLA_DEV_QPOS_RANGE);
    pos0 = pos0 < 0 ? 0 : a.max_len - a.T;
  }
  it.nq = min(TQ, a.T - it.q0);
  it.qp0 = pos0 + it.q0;
  it.qp_last = it.qp0 + it.nq - 1;
  it.nk = it.qp_last / TK + 1;
  return it;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    mha_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_kr,
                  const MhaArgs a, const int ctr) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Ctl ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int items = ((a.T + TQ - 1) / TQ) * a.n_h * a.B;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NKS; ++i) { mbar_init(&ctl.k_full[i], 1); mbar_init(&ctl.k_empty[i], 1); }
    for (int i = 0; i < NVS; ++i) { mbar_init(&ctl.v_full[i], 1); mbar_init(&ctl.v_empty[i], 1); }
    mbar_init(&ctl.q_ready, 8);
    mbar_init(&ctl.s_full, 1);
    mbar_init(&ctl.s_free, 8);
    mbar_init(&ctl.p_full, 8);
    mbar_init(&ctl.pv_done, 1);
    mbar_init(&ctl.mma_done, 2);
    for (int i = 0; i < NIR; ++i) { mbar_init(&ctl.ir_full[i], 1); mbar_init(&ctl.ir_empty[i], IR_READERS); }
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
  const uint32_t sbase = smem_u32(smem);
  // The e-th item of this CTA (-1: no more), from the item ring; each reading
  // thread (one per reading warp) frees its entry once it has the index.
  auto next_item = [&](int e, int& k) -> bool {
    const int sl = e % NIR;
    if (!wait_or_abort(&ctl.ir_full[sl], (e / NIR) & 1, ctl, a.status)) return false;
    k = *reinterpret_cast<volatile int*>(&ctl.ir_item[sl]);
    mbar_arrive(&ctl.ir_empty[sl]);
    return true;
  };

  // The key ring carries, per item, the query tile (3 chunks, the size of a
  // key stage) and then the item's key tiles; load n of the CTA goes to stage
  // n % NKS. The value ring and the score / P / PV handshakes count the CTA's
  // key tiles over all its items.
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producers
    // lane 0: the queries and the key stages; lane 1: the value stages
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_kr);
      int n = 0;
      bool ok = true;
      for (int e = 0; ok; ++e) {
        const int sl = e % NIR;
        if (e >= NIR) ok = wait_or_abort(&ctl.ir_empty[sl], ((e / NIR) - 1) & 1, ctl, a.status);
        if (!ok) break;
        const unsigned int got = atomicAdd(&g_item_next[ctr], 1u);
        const int k = got < (unsigned int)items ? (int)got : -1;
        ctl.ir_item[sl] = k;
        mbar_arrive(&ctl.ir_full[sl]);
        if (k < 0) break;
        const Item it = item_of(a, k, false);
        for (int j = -1; j < it.nk; ++j, ++n) {   // j = -1: the query tile
          const int st = n % NKS;
          if (n >= NKS) ok = wait_or_abort(&ctl.k_empty[st], ((n / NKS) - 1) & 1, ctl, a.status);
          if (!ok) break;
          uint8_t* dst = smem + KRING_OFF + st * KSTAGE;
          mbar_arrive_expect_tx(&ctl.k_full[st], KSTAGE);
          if (j < 0) {
            tma_load_3d(dst, &map_q, &ctl.k_full[st], 0, it.b * a.T + it.q0, it.head * 3);
          } else {
            const int krow = it.b * a.max_len + j * TK;
            tma_load_3d(dst, &map_k, &ctl.k_full[st], 0, krow, it.head * 2);
            tma_load_2d(dst + 2 * CHUNK, &map_kr, &ctl.k_full[st], 0, krow);
          }
        }
      }
      if (!ok) drain_ring(ctl.k_full, NKS, n);   // no copy lands after the CTA moves on
    } else if (lane == 1) {
      prefetch_tensormap(&map_v);
      int n = 0, k = 0;
      bool ok = true;
      for (int e = 0; ok && (ok = next_item(e, k)) && k >= 0; ++e) {
        const Item it = item_of(a, k, false);
        for (int j = 0; j < it.nk; ++j, ++n) {
          const int st = n % NVS;
          if (n >= NVS) ok = wait_or_abort(&ctl.v_empty[st], ((n / NVS) - 1) & 1, ctl, a.status);
          if (!ok) break;
          mbar_arrive_expect_tx(&ctl.v_full[st], VSTAGE);
          tma_load_3d(smem + VRING_OFF + st * VSTAGE, &map_v, &ctl.v_full[st], 0, it.b * a.max_len + j * TK,
                      it.head * 2);
        }
      }
      if (!ok) drain_ring(ctl.v_full, NVS, n);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK issuer
    // S(g) = Q . K(g)^T (Q from TMEM) once key stage g has landed and the
    // softmax has read S(g-1); for an item's first tile, once its queries are
    // in TMEM (which also frees their stage). QK and PV have an issuing thread
    // each, so that a PV never waits behind the next tile's load.
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16(TQ, TK, false, false);
      const uint64_t k_desc = sdesc_sw128(sbase + KRING_OFF, 16, 1024);
      int n = 0, g = 0, k = 0;
      bool ok = true;
      for (int i = 0; ok && (ok = next_item(i, k)) && k >= 0; ++i) {
        const Item it = item_of(a, k, false);
        ok = wait_or_abort(&ctl.q_ready, i & 1, ctl, a.status);
        if (!ok) break;
        mbar_arrive(&ctl.k_empty[n % NKS]);   // the query stage: copied into TMEM
        ++n;
        for (int j = 0; j < it.nk; ++j, ++n, ++g) {
          const int st = n % NKS;
          ok = wait_or_abort(&ctl.k_full[st], (n / NKS) & 1, ctl, a.status) &&
               (g < 1 || wait_or_abort(&ctl.s_free, (g - 1) & 1, ctl, a.status));
          if (!ok) break;
          tc_fence_after();
          const uint64_t kd = k_desc + (uint64_t)((st * KSTAGE) >> 4);
#pragma unroll
          for (int c = 0; c < 3; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ta(tbase + S_COL, tbase + Q_COL + c * 32 + kk * 8, kd + (uint64_t)((c * CHUNK + kk * 32) >> 4),
                          IDESC_QK, (c > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&ctl.s_full);
          mma_commit(&ctl.k_empty[st]);   // the key stage: its QK is done
        }
      }
      // nothing of this CTA's reaches the tensor cores after it moves on
      mma_commit(&ctl.mma_done);
      mbar_wait(&ctl.mma_done, 0, WAIT_CYCLES / 8);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ PV issuer
    // O += P(g) . V(g) once the softmax has written P(g) and V(g) has landed;
    // an item's first PV starts O afresh. The value stage is free when this
    // PV completes.
    if (lane == 0) {
      constexpr uint32_t IDESC_PV = idesc_bf16(TQ, DH, false, true);
      const uint64_t v_desc = sdesc_sw128(sbase + VRING_OFF, CHUNK, 1024);
      int g = 0, k = 0;
      bool ok = true;
      for (int e = 0; ok && (ok = next_item(e, k)) && k >= 0; ++e) {
        const Item it = item_of(a, k, false);
        for (int j = 0; j < it.nk; ++j, ++g) {
          const int st = g % NVS;
          ok = wait_or_abort(&ctl.p_full, g & 1, ctl, a.status) &&
               wait_or_abort(&ctl.v_full[st], (g / NVS) & 1, ctl, a.status);
          if (!ok) break;
          tc_fence_after();
          const uint64_t vd = v_desc + (uint64_t)((st * VSTAGE) >> 4);
#pragma unroll
          for (int kk = 0; kk < TK / 16; ++kk)
            mma_bf16_ta(tbase + O_COL, tbase + P_COL + kk * 8, vd + (uint64_t)((kk * 2048) >> 4), IDESC_PV,
                        (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&ctl.pv_done);
          mma_commit(&ctl.v_empty[st]);
        }
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
    const float sl2 = a.scale_log2;
    constexpr int HK = TK / 2;                         // keys per half
    // An item's query tile from its key-ring stage into TMEM (row r = lane r,
    // 32 columns per 64-column chunk): half 0 moves chunks 0 and 1, half 1
    // chunk 2. The previous item's last QK, the last reader of the queries in
    // TMEM, has completed: its scores have been waited for.
    auto move_queries = [&](int n) -> bool {
      const int st = n % NKS;
      if (!pair_all(quarter, __all_sync(0xffffffffu, wait_or_abort(&ctl.k_full[st], (n / NKS) & 1, ctl, a.status))))
        return false;
      const uint8_t* qs = smem + KRING_OFF + st * KSTAGE + (r >> 3) * 1024 + (r & 7) * 128;
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
      if (lane == 0) mbar_arrive(&ctl.q_ready);
      return true;
    };
    // the CTA's items, read by lane 0 of each softmax warp
    auto item_at = [&](int e, int& k) -> bool {
      int kk = 0;
      bool got = true;
      if (lane == 0) got = next_item(e, kk);
      got = pair_all(quarter, __all_sync(0xffffffffu, __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0));
      k = __shfl_sync(0xffffffffu, kk, 0);
      return got;
    };
    int n = 0, g = 0;   // key-ring loads and key tiles of this CTA so far
    int k = 0, k_next = 0;
    bool ok = item_at(0, k) && (k < 0 || move_queries(0));
    Item nxt = item_of(a, k < 0 ? 0 : k, threadIdx.x == 96 && k >= 0);
    for (int e = 0; ok && k >= 0; ++e, k = k_next) {
      const Item it = nxt;
      const int qp = it.qp0 + r;                       // this row's position (rows past nq: not stored)
      float m_ref = -INFINITY, l = 0.f;
      ++n;                                             // past the query tile
      for (int j = 0; j < it.nk && ok; ++j, ++n, ++g) {
        const int k0 = j * TK + half * HK;
        ok = pair_all(quarter, __all_sync(0xffffffffu, wait_or_abort(&ctl.s_full, g & 1, ctl, a.status)));
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
        ctl.mx[g & 1][half][r] = mx;
        pair_sync(quarter);
        mx = fmaxf(mx, ctl.mx[g & 1][half ^ 1][r]);   // the row's tile maximum, the same in both halves
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
        // P(g) replaces P(g-1) in TMEM and O is rescaled: both only after
        // PV(g-1) (for an item's first tile, the previous item's epilogue
        // already waited for its last PV)
        if (j > 0) {
          ok = pair_all(quarter, __all_sync(0xffffffffu, wait_or_abort(&ctl.pv_done, (g - 1) & 1, ctl, a.status)));
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
        if (j == it.nk - 1 && it.qp_last - j * TK + 1 < TK) {
          const int st = g % NVS;
          ok = pair_all(quarter, __all_sync(0xffffffffu, wait_or_abort(&ctl.v_full[st], (g / NVS) & 1, ctl, a.status)));
          if (!ok) break;
          const int first = it.qp_last - j * TK + 1;   // rows first .. TK-1 of both v_C chunks
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
      if (!ok) break;
      // The next item's queries go into TMEM now, so that its first QK runs
      // while this item's last PV and epilogue do.
      ok = item_at(e + 1, k_next) && (k_next < 0 || move_queries(n));
      if (ok && k_next >= 0) nxt = item_of(a, k_next, threadIdx.x == 96);   // its position is read during the epilogue
      // ---------------------------------------------------------------- epilogue
      if (ok) ok = pair_all(quarter, __all_sync(0xffffffffu, wait_or_abort(&ctl.pv_done, (g - 1) & 1, ctl, a.status)));
      if (!ok) break;
      ctl.ls[half][r] = l;
      pair_sync(quarter);
      l += ctl.ls[half ^ 1][r];
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool store = r < it.nq;
      __nv_bfloat16* orow =
          static_cast<__nv_bfloat16*>(a.o) + (((size_t)it.b * a.T + it.q0 + r) * a.n_h + it.head) * DH;
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
      if (store && half == 0) a.lse[((size_t)it.b * a.T + it.q0 + r) * a.n_h + it.head] = (m_ref + log2f(l)) * kLn2;
      // the O reads are done before this item's successor writes P (program
      // order) and its first PV starts O afresh; the sums' exchange slots are
      // rewritten only after the next pair_sync
      tc_fence_before();
      pair_sync(quarter);
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, TMEM_COLS);
  // The last CTA to leave resets the launch's counters (every CTA has taken
  // its last index by now) for the next launch that uses them.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&g_cta_done[ctr], 1u) == gridDim.x - 1) {
      atomicExch(&g_item_next[ctr], 0u);
      atomicExch(&g_cta_done[ctr], 0u);
      __threadfence();
    }
  }
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
  // one CTA per SM (or per item, when there are fewer items)
  static int sms = 0;
  if (sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return cudaErrorInvalidValue;
  }
  const long long items = (long long)((a.T + TQ - 1) / TQ) * a.n_h * a.B;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  LaunchCfg lc(dim3((unsigned)(items < sms ? items : sms)), dim3(NTHREADS), SMEM_DYN, s);
  // each launch in a stream's flight uses counters of its own (slots rotate)
  static std::atomic<unsigned int> next_ctr{0};
  const int ctr = (int)(next_ctr.fetch_add(1u) % NCTR);
  cudaError_t e = cudaLaunchKernelEx(&lc.cfg, mha_tc_kernel, map_q, map_k, map_v, map_kr, a, ctr);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
