// Tensor-core split-KV latent attention for layers with few heads (n_h <= 16;
// d_c = 128, d_r = 32 or 64, bf16), where the step is purely bound by
// reading the cache: 320 bytes per cached row against 2 n_h (d_c + d_r + d_c)
// FLOPs, about 15 FLOP/B for 8 heads.
//
// What is computed (page "MLA：潜在表示压缩与解耦 RoPE", §6 two-part score and
// §7 softmax with scale 1/sqrt(d_h + d_r); page "Latent 压缩", value deferral):
// for every head i of every sequence
//   s_{i,t} = q_abs_i . row_t * scale,  o_lat_i = sum_t softmax_t(s_{i,t}) c_KV_t,  and the LSE.
//
// With a handful of heads, the heads cannot fill the 128-row side of a
// tcgen05 MMA, so both products are transposed and the cache rows take it:
//   S^T = C . Q^T      M = 128 cache rows, N = 16 (the heads, padded), K = d_c + d_r
//   O_t^T = V^T . P^T  M = 128 latent columns (per block), N = 16, K = the tile's rows
// Both read the same TMA-fed shared-memory tile: QK as a K-major operand,
// PV as an MN-major one. The fp32 results live in TMEM (16 columns each);
// the softmax threads own one cache row (S) and one latent column (O) each.
// O_t is the tile's unnormalised contribution; the threads fold it into an
// fp32 accumulator in registers, O = O * alpha + O_t, so TMEM never needs a
// rescale and every MMA starts from zero.
//
// One CTA per SM streams its chunk of the plan (one whole sequence, or an
// equal share of all sequences' rows laid end to end, as for every decode
// kernel here) through a ring of 128-row tiles: the latent part as one box of d_c/64 chunks of
// 64 columns (128-byte swizzle), the RoPE part as one box of its own
// (64- or 128-byte swizzle). Warp 0 issues TMA, warp 1 the QK MMAs, warp 2
// the PV MMAs, and groups of four warps from warp 3 on run the online
// softmax for four heads each (base 2, lazy
// reference maximum as in the many-head kernel: it moves only when a tile's
// maximum rises more than 8 above it), write P, and fold O. A piece that
// covers a whole sequence writes o_lat/lse, any other piece a partial slot
// that the LSE combine kernel merges.
//
// Every mbarrier wait is bounded; on expiry the CTA records MLA_DEV_TIMEOUT,
// stops issuing work, waits (bounded) for its own copies in flight and frees
// its TMEM.
#include "decode_narrow.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int TR = 128;                  // cache rows per tile (MMA M of QK)
constexpr int NPAD = 16;                 // heads padded to the MMA's N
constexpr int HPG = 4;                   // heads per softmax warp group (4 warps, one per TMEM lane quarter)
constexpr long long WAIT_CYCLES = 4000000000LL;  // ~2 s
constexpr float kLn2 = 0.693147180559945309f;
constexpr float RESCALE_THRESHOLD = 8.0f;
constexpr int SMEM_LIMIT = 227 * 1024;    // opt-in shared memory per CTA
constexpr int CTL_RESERVE = 2048;         // the static control block (Ctl), rounded up
constexpr int MAX_SLOTS = 6;
constexpr int NSB = 4;                   // S^T buffers in TMEM
constexpr int NPP = 3;                   // P^T buffers in shared memory
constexpr int NOB = 4;                   // O_t^T buffers in TMEM
constexpr int FOLD = 2;                  // the softmax folds O_t of tile g - FOLD while at tile g
static_assert(NPP >= FOLD + 1, "a P buffer is rewritten only after the PV that read it was folded");

// Shared-memory descriptor with an explicit layout type (the 3-bit field at
// bit 61): 2 = 128-byte swizzle, 4 = 64-byte swizzle. Addresses in bytes.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

template <int DC, int DR>
struct Shape {
  static constexpr int NCL = DC / 64;                 // latent column chunks
  static constexpr int NB = DC / 128;                 // 128-column latent blocks (PV M)
  static constexpr int LAT_CHUNK = TR * 128;          // 16 KB: 128 rows x 64 columns
  static constexpr int ROPE_ROW = DR * 2;             // bytes of one row's RoPE part
  static constexpr int ROPE_BYTES = TR * ROPE_ROW;
  static constexpr int SLOT = NCL * LAT_CHUNK + ROPE_BYTES;
  static constexpr uint32_t ROPE_LAYOUT = DR == 64 ? 2u : 4u;   // 128- or 64-byte swizzle
  static constexpr int ROPE_SBO = 8 * ROPE_ROW;
  // Q (B operand of QK, K-major): [NCL chunks][16 rows][128 B], then the RoPE part [16 rows][ROPE_ROW]
  static constexpr int QL_CHUNK = NPAD * 128;         // 2 KB
  static constexpr int Q_BYTES = NCL * QL_CHUNK + NPAD * ROPE_ROW;
  static constexpr int Q_STRIDE = (Q_BYTES + 1023) / 1024 * 1024;
  // P^T (B operand of PV, K-major): [2 chunks of 64 rows][16 heads][128 B]
  static constexpr int P_BYTES = 2 * NPAD * 128;      // 4 KB
  // as many ring slots as the rest leaves room for: the ring's depth is what
  // hides the HBM latency at one CTA per SM
  static constexpr int RING_BUDGET = SMEM_LIMIT - 1024 - 2 * Q_STRIDE - NPP * P_BYTES - CTL_RESERVE;
  static constexpr int NSLOT = (RING_BUDGET / SLOT) < MAX_SLOTS ? (RING_BUDGET / SLOT) : MAX_SLOTS;
  static constexpr int RING_OFF = 0;
  static constexpr int Q_OFF = NSLOT * SLOT;           // two query buffers (piece parity)
  static constexpr int P_OFF = Q_OFF + 2 * Q_STRIDE;   // NPP P buffers (tile g in g % NPP)
  static constexpr int END = P_OFF + NPP * P_BYTES;
  // the split plan when the kernel computes it (B + PLAN_EXTRA entries): what the ring leaves, at most 4 KB
  static constexpr int PLAN_OFF = END;
  static constexpr int PLAN_ROOM = (SMEM_LIMIT - CTL_RESERVE - 1024 - END) / 16 * 16;
  static constexpr int PLAN_BYTES = PLAN_ROOM < 4096 ? PLAN_ROOM : 4096;
  static constexpr int SMEM_DYN = END + PLAN_BYTES + 1024;
  // TMEM: NSB S^T buffers (16 columns each), then NOB O_t^T buffers (16 per latent block)
  static constexpr uint32_t S_COL = 0;
  static constexpr uint32_t O_COL = NSB * NPAD;
  static constexpr uint32_t TMEM_USED = O_COL + NOB * NB * NPAD;
  static constexpr uint32_t TMEM_COLS = TMEM_USED <= 64 ? 64 : (TMEM_USED <= 128 ? 128 : 256);
  static_assert(DC % 128 == 0 && DC <= 256, "latent width");
  static_assert(DR == 32 || DR == 64, "RoPE width");
  static_assert(NSLOT >= 3, "ring");
  static_assert(SLOT % 1024 == 0, "slot alignment");
  static_assert(SMEM_DYN + CTL_RESERVE <= SMEM_LIMIT, "shared memory");
  static_assert(PLAN_BYTES >= 256, "plan room");
};

struct Ctl {   // static shared memory: at most CTL_RESERVE bytes
  uint64_t full[MAX_SLOTS], empty[MAX_SLOTS];
  uint64_t q_full[2], q_free[2];
  uint64_t s_full[NSB], s_free[NSB];
  uint64_t p_full[NPP];
  uint64_t o_full[NOB], o_free[NOB];
  uint32_t tmem_base;
  int abort;
  long long wait_limit;       // cycles before a wait gives up
  uint64_t mma_done;          // every MMA of both issuers has completed (two arrivals)
  float wmax[2][4][NPAD];     // per tile parity, TMEM lane quarter and head: the tile's maximum
  float wsum[4][NPAD];        // per TMEM lane quarter and head: the piece's softmax sum
};
static_assert(sizeof(Ctl) + 512 <= CTL_RESERVE, "control block and the plan's scratch");

// Every wait gives up after ctl.wait_limit cycles, or as soon as another role
// of this CTA has given up; the first to expire records MLA_DEV_TIMEOUT.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Ctl& ctl, int32_t* status) {
  volatile int* ab = reinterpret_cast<volatile int*>(&ctl.abort);
  if (*ab) return false;
  if (mbar_wait_abortable(bar, parity, ctl.wait_limit, ab)) return true;
  if (!*ab) atomicOr(status, MLA_DEV_TIMEOUT);
  *ab = 1;
  return false;
}

// Named barriers of softmax group grp (ids 1 .. 4, 128 threads each).
__device__ __forceinline__ void grp_bar(int grp) { asm volatile("bar.sync %0, 128;" ::"r"(1 + grp) : "memory"); }
__device__ __forceinline__ bool grp_any(int grp, bool v) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n barrier.cta.red.or.pred po, %2, 128, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(1 + grp)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ int find_seq_n(const int32_t* __restrict__ cum, int B, int r) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cum[mid] <= r) lo = mid; else hi = mid;
  }
  while (lo < B - 1 && cum[lo + 1] <= r) ++lo;
  return lo;
}

// The pieces (sequence, row range) of one chunk of the plan.
struct Pieces {
  const int32_t* cum; int B, start, end, b;
  __device__ void init(const int32_t* c, int B_, int chunk) {
    cum = c; B = B_;
    if (cum[B + 3]) {
      b = chunk < B ? chunk : B;
      start = chunk < B ? cum[chunk] : 0;
      end = chunk < B ? cum[chunk + 1] : 0;
      return;
    }
    const int cl = cum[B + 1], total = cum[B + 2];
    start = chunk * cl;
    end = min(start + cl, total);
    b = start < end ? find_seq_n(cum, B, start) : B;
  }
  __device__ bool next(int& seq, int& t0, int& t1, bool& whole) {
    while (b < B && cum[b] < end) {
      const int s0 = cum[b], s1 = cum[b + 1];
      const int cur = b++;
      if (s1 == s0) continue;
      const int p0 = max(s0, start), p1 = min(s1, end);
      seq = cur; t0 = p0 - s0; t1 = p1 - s0; whole = (p0 == s0 && p1 == s1);
      return true;
    }
    return false;
  }
};

__device__ __forceinline__ void drain_ring(uint64_t* full, int ring, int issued) {
  for (int s = 0; s < ring; ++s) {
    if (issued <= s) break;
    const int last = s + ring * ((issued - 1 - s) / ring);
    mbar_wait(&full[s], (uint32_t)((last / ring) & 1), WAIT_CYCLES / 8);
  }
}

// NGRP softmax groups of 4 warps, each owning HPG heads (n_h <= HPG * NGRP).
template <int DC, int DR, int NGRP>
__global__ void __launch_bounds__(96 + 128 * NGRP, 1)
    decode_narrow_kernel(const __grid_constant__ CUtensorMap map_lat, const __grid_constant__ CUtensorMap map_rope,
                         const __grid_constant__ CUtensorMap map_qlat, const __grid_constant__ CUtensorMap map_qrope,
                         const DecodeArgs a) {
  using L = Shape<DC, DR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Ctl ctl;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x;
  const int B = a.B, n_h = a.n_h;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::NSLOT; ++i) { mbar_init(&ctl.full[i], 1); mbar_init(&ctl.empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&ctl.q_full[i], 1); mbar_init(&ctl.q_free[i], 1); }
    for (int i = 0; i < NSB; ++i) { mbar_init(&ctl.s_full[i], 1); mbar_init(&ctl.s_free[i], 4 * NGRP); }
    for (int i = 0; i < NPP; ++i) mbar_init(&ctl.p_full[i], 4 * NGRP);
    for (int i = 0; i < NOB; ++i) { mbar_init(&ctl.o_full[i], 1); mbar_init(&ctl.o_free[i], 4 * NGRP); }
    mbar_init(&ctl.mma_done, 2);
    ctl.abort = 0;
    ctl.wait_limit = a.wait_cycles > 0 ? a.wait_cycles : WAIT_CYCLES;
    fence_mbar_init();
  }
  // The padded head rows of Q and P feed only score / output columns that are
  // never read; zero them once so that no stale bits reach the tensor cores.
  for (int i = threadIdx.x * 16; i < 2 * L::Q_STRIDE + NPP * L::P_BYTES; i += (96 + 128 * NGRP) * 16)
    *reinterpret_cast<uint4*>(smem + L::Q_OFF + i) = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl.tmem_base;
  pdl_trigger();
  pdl_wait();      // the plan, the queries and the cache come from earlier kernels
  const uint32_t sbase = smem_u32(smem);
  // The split plan: every CTA works it out from the lengths (CTA 0 also
  // stores it for the merge kernel), or it comes from the plan launch.
  const int32_t* plan = a.plan;
  if (a.inline_plan) {
    int32_t* ps = reinterpret_cast<int32_t*>(smem + L::PLAN_OFF);
    plan_rows(a.seqlens, B, a.max_len, a.grid_chunks, 64, a.allow_whole, 2 * TR, ps, a.status, blockIdx.x == 0);
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i < B + PLAN_EXTRA; i += 96 + 128 * NGRP) a.plan[i] = ps[i];
    plan = ps;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&map_lat);
      prefetch_tensormap(&map_rope);
      prefetch_tensormap(&map_qlat);
      prefetch_tensormap(&map_qrope);
      Pieces it;
      it.init(plan, B, chunk);
      int seq, t0, t1;
      bool whole;
      int i = 0, piece = 0, qissued = 0;
      bool ok = true;
      while (ok && it.next(seq, t0, t1, whole)) {
        const int qb = piece & 1;
        if (piece >= 2) ok = wait_or_abort(&ctl.q_free[qb], ((piece >> 1) - 1) & 1, ctl, a.status);
        if (!ok) break;
        uint8_t* qs = smem + L::Q_OFF + qb * L::Q_STRIDE;
        mbar_arrive_expect_tx(&ctl.q_full[qb], (uint32_t)(n_h * (DC * 2 + DR * 2)));
        for (int c = 0; c < L::NCL; ++c) tma_load_2d(qs + c * L::QL_CHUNK, &map_qlat, &ctl.q_full[qb], c * 64, seq * n_h);
        tma_load_2d(qs + L::NCL * L::QL_CHUNK, &map_qrope, &ctl.q_full[qb], 0, seq * n_h);
        ++qissued;
        for (int r = t0; r < t1; r += TR, ++i) {
          const int sl = i % L::NSLOT;
          if (i >= L::NSLOT) ok = wait_or_abort(&ctl.empty[sl], ((i / L::NSLOT) - 1) & 1, ctl, a.status);
          if (!ok) break;
          uint8_t* dst = smem + L::RING_OFF + sl * L::SLOT;
          const int row = seq * a.max_len + r;
          mbar_arrive_expect_tx(&ctl.full[sl], (uint32_t)L::SLOT);
          tma_load_3d(dst, &map_lat, &ctl.full[sl], 0, row, 0);
          tma_load_2d(dst + L::NCL * L::LAT_CHUNK, &map_rope, &ctl.full[sl], 0, row);
        }
        ++piece;
      }
      if (!ok) {   // no copy lands after the CTA moves on
        drain_ring(ctl.full, L::NSLOT, i);
        drain_ring(ctl.q_full, 2, qissued);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK issuer
    // S^T of tile g into TMEM buffer g % NSB as soon as the tile has landed
    // and the softmax has read the buffer's previous tile. QK and PV have an
    // issuing thread each: a small-N MMA costs its issuing thread about as
    // long as the tensor core takes to run it, so one thread alone would
    // leave the tensor core idle between the two streams.
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16(128, NPAD, false, false);
      // descriptors built once; each MMA adds a byte offset (>> 4) to the start address field
      const uint64_t ring_k = sdesc(sbase + L::RING_OFF, 16, 1024, 2);
      const uint64_t ring_r = sdesc(sbase + L::RING_OFF, 16, L::ROPE_SBO, L::ROPE_LAYOUT);
      const uint64_t q_k = sdesc(sbase + L::Q_OFF, 16, 1024, 2);
      const uint64_t q_r = sdesc(sbase + L::Q_OFF, 16, L::ROPE_SBO, L::ROPE_LAYOUT);
      Pieces it;
      it.init(plan, B, chunk);
      int seq, t0, t1;
      bool whole;
      int piece = 0, g = 0;
      bool ok = true;
      while (ok && it.next(seq, t0, t1, whole)) {
        const int qb = piece & 1;
        ok = wait_or_abort(&ctl.q_full[qb], (piece >> 1) & 1, ctl, a.status);
        for (int r = t0; r < t1 && ok; r += TR, ++g) {
          const int sl = g % L::NSLOT, sb = g % NSB;
          ok = wait_or_abort(&ctl.full[sl], (g / L::NSLOT) & 1, ctl, a.status) &&
               (g < NSB || wait_or_abort(&ctl.s_free[sb], ((g / NSB) - 1) & 1, ctl, a.status));
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tbase + L::S_COL + sb * NPAD;
          const uint64_t a0 = ring_k + (uint64_t)((sl * L::SLOT) >> 4);
          const uint64_t b0 = q_k + (uint64_t)((qb * L::Q_STRIDE) >> 4);
          // S^T = C . Q^T over the latent chunks, then the RoPE part
#pragma unroll
          for (int c = 0; c < L::NCL; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16(d, a0 + (uint64_t)((c * L::LAT_CHUNK + k * 32) >> 4),
                       b0 + (uint64_t)((c * L::QL_CHUNK + k * 32) >> 4), IDESC_QK, (c > 0 || k > 0) ? 1u : 0u);
          const uint64_t ar = ring_r + (uint64_t)((sl * L::SLOT + L::NCL * L::LAT_CHUNK) >> 4);
          const uint64_t br = q_r + (uint64_t)((qb * L::Q_STRIDE + L::NCL * L::QL_CHUNK) >> 4);
#pragma unroll
          for (int k = 0; k < DR / 16; ++k)
            mma_bf16(d, ar + (uint64_t)((k * 32) >> 4), br + (uint64_t)((k * 32) >> 4), IDESC_QK, 1u);
          mma_commit(&ctl.s_full[sb]);
        }
        // the piece's last QK: its query buffer may be refilled
        if (ok) mma_commit(&ctl.q_free[qb]);
        ++piece;
      }
      // nothing of this CTA's reaches the tensor cores after it moves on
      mma_commit(&ctl.mma_done);
      mbar_wait(&ctl.mma_done, 0, WAIT_CYCLES / 8);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ PV issuer
    // O_t^T of tile g into TMEM buffer g % NOB once the softmax has written
    // P^T(g) and folded the buffer's previous tile; the tile's ring slot is
    // released when this PV completes (its QK completed before P existed).
    if (lane == 0) {
      constexpr uint32_t IDESC_PV = idesc_bf16(128, NPAD, true, false);
      const uint64_t ring_v = sdesc(sbase + L::RING_OFF, L::LAT_CHUNK, 1024, 2);
      const uint64_t p_k = sdesc(sbase + L::P_OFF, 16, 1024, 2);
      Pieces it;
      it.init(plan, B, chunk);
      int seq, t0, t1;
      bool whole;
      int g = 0;
      bool ok = true;
      while (ok && it.next(seq, t0, t1, whole)) {
        for (int r = t0; r < t1 && ok; r += TR, ++g) {
          const int pb = g % NPP, ob = g % NOB, sl = g % L::NSLOT;
          ok = wait_or_abort(&ctl.p_full[pb], (g / NPP) & 1, ctl, a.status) &&
               (g < NOB || wait_or_abort(&ctl.o_free[ob], ((g / NOB) - 1) & 1, ctl, a.status));
          if (!ok) break;
          tc_fence_after();
          // O_t^T[ob] = V^T . P^T over the tile's valid rows, 16 per MMA
          const int ksteps = (min(TR, t1 - r) + 15) >> 4;
          const uint64_t a0 = ring_v + (uint64_t)((sl * L::SLOT) >> 4);
          const uint64_t b0 = p_k + (uint64_t)((pb * L::P_BYTES) >> 4);
#pragma unroll
          for (int mb = 0; mb < L::NB; ++mb) {
            const uint32_t d = tbase + L::O_COL + (uint32_t)(ob * L::NB + mb) * NPAD;
#pragma unroll
            for (int kk = 0; kk < TR / 16; ++kk)
              if (kk < ksteps)
                mma_bf16(d, a0 + (uint64_t)((mb * 2 * L::LAT_CHUNK + kk * 16 * 128) >> 4),
                         b0 + (uint64_t)(((kk >> 2) * (NPAD * 128) + (kk & 3) * 32) >> 4), IDESC_PV,
                         kk > 0 ? 1u : 0u);
          }
          mma_commit(&ctl.o_full[ob]);
          mma_commit(&ctl.empty[sl]);   // the tile's slot: its QK and PV are done
        }
      }
      mma_commit(&ctl.mma_done);
      mbar_wait(&ctl.mma_done, 0, WAIT_CYCLES / 8);
    }
  } else {
    // ------------------------------------------------------------ softmax warps 3 .. 2 + 4 NGRP
    // Group grp (warps 3+4grp .. 6+4grp) owns heads h0 .. h0+3: the online
    // softmax of different heads shares nothing, so each group keeps its own
    // running maxima, sums and O columns and meets only its own four warps.
    const int grp = (warp - 3) >> 2;
    const int h0 = grp * HPG;
    const int quarter = warp & 3;
    const int t = quarter * 32 + lane;                // TMEM lane: cache row of S, latent column of O
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = a.scale_log2;
    Pieces it;
    it.init(plan, B, chunk);
    int seq, t0, t1;
    bool whole;
    int g = 0;
    bool ok = true;
    // o_acc: this thread's latent column(s) of O for the group's heads; hist:
    // the rescale factors of the tiles whose O_t is not folded in yet
    float m_ref[HPG], l_part[HPG], o_acc[L::NB][HPG], hist[FOLD][HPG];
    // Fold O_t of tile gp into the accumulator: O = O * alpha(gp) + O_t.
    auto fold = [&](int gp, const float (&al)[HPG]) -> bool {
      const int ob = gp % NOB;
      // warp-uniform: the TMEM loads below are warp-collective
      const bool w = __all_sync(0xffffffffu, wait_or_abort(&ctl.o_full[ob], (gp / NOB) & 1, ctl, a.status));
      if (!w) return false;
      tc_fence_after();
#pragma unroll
      for (int mb = 0; mb < L::NB; ++mb) {
        float v[4];
        tmem_ld4(tbase + lane_base + L::O_COL + (uint32_t)(ob * L::NB + mb) * NPAD + h0, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < HPG; ++j) o_acc[mb][j] = fmaf(o_acc[mb][j], al[j], v[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.o_free[ob]);
      return true;
    };
    while (ok && it.next(seq, t0, t1, whole)) {
      const int ntiles = (t1 - t0 + TR - 1) / TR;
      const int g0 = g;                               // the piece's first tile
#pragma unroll
      for (int j = 0; j < HPG; ++j) {
        m_ref[j] = -INFINITY; l_part[j] = 0.f;
#pragma unroll
        for (int mb = 0; mb < L::NB; ++mb) o_acc[mb][j] = 0.f;
      }
      for (int k = 0; k < ntiles; ++k, ++g) {
        const int nvalid = min(TR, t1 - t0 - k * TR);
        const int sb = g % NSB;
        const bool w = __all_sync(0xffffffffu, wait_or_abort(&ctl.s_full[sb], (g / NSB) & 1, ctl, a.status));
        float s[HPG];
        if (w) {
          tc_fence_after();
          tmem_ld4(tbase + lane_base + L::S_COL + sb * NPAD + h0, s);
          tmem_ld_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && w) mbar_arrive(&ctl.s_free[sb]);
        const bool valid = t < nvalid;
        // scaled scores in base 2 (rows past the piece end and absent heads at -inf)
        bool rise = false;
#pragma unroll
        for (int j = 0; j < HPG; ++j) {
          s[j] = (valid && h0 + j < n_h) ? s[j] * sl2 : -INFINITY;
          rise |= s[j] > m_ref[j] + RESCALE_THRESHOLD;
        }
        // The reference maxima move only when some score of the group rises
        // more than the threshold above them (always on a piece's first tile);
        // otherwise the tile needs no reduction at all.
        const bool stop = !w || !ok;
        rise = grp_any(grp, rise || stop);
        if (rise && grp_any(grp, stop)) { ok = false; break; }   // every warp of the group leaves together
        float alpha[HPG];
#pragma unroll
        for (int j = 0; j < HPG; ++j) alpha[j] = 1.f;
        if (rise) {
          const int mx = g & 1;
#pragma unroll
          for (int j = 0; j < HPG; ++j) {
            float m = s[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) ctl.wmax[mx][quarter][h0 + j] = m;
          }
          grp_bar(grp);
#pragma unroll
          for (int j = 0; j < HPG; ++j) {
            const int hh = h0 + j;
            if (hh >= n_h) continue;
            const float mt = fmaxf(fmaxf(ctl.wmax[mx][0][hh], ctl.wmax[mx][1][hh]),
                                   fmaxf(ctl.wmax[mx][2][hh], ctl.wmax[mx][3][hh]));
            if (m_ref[j] == -INFINITY || mt > m_ref[j] + RESCALE_THRESHOLD) {
              alpha[j] = (m_ref[j] == -INFINITY) ? 0.f : ex2_approx(m_ref[j] - mt);
              m_ref[j] = mt;
            }
          }
        }
        // P^T row t of this tile for the group's heads: one bf16 value per head,
        // in the K-major layout [row / 64][head][128 B] (128-byte swizzle). The
        // buffer's last reader, PV of tile g - NPP, was folded in at least one
        // tile ago.
        uint8_t* pbuf = smem + L::P_OFF + (g % NPP) * L::P_BYTES;
        {
          const int rr = t & 63;
          uint8_t* base = pbuf + (t >> 6) * (NPAD * 128) + (rr & 7) * 2;
#pragma unroll
          for (int j = 0; j < HPG; ++j) {
            const int hh = h0 + j;
            if (hh >= n_h) break;   // absent heads keep the zeros written at start
            const float p = ex2_approx(s[j] - m_ref[j]);   // 0 for masked rows
            l_part[j] = fmaf(l_part[j], alpha[j], p);
            *reinterpret_cast<__nv_bfloat16*>(base + (hh >> 3) * 1024 + (hh & 7) * 128 + (((rr >> 3) ^ (hh & 7)) << 4)) =
                __float2bfloat16_rn(p);
          }
        }
        // The tile's rows past the piece end inside its last 16-row MMA step
        // may hold anything (even NaN): zero their latent part before PV reads it.
        if (grp == 0 && nvalid < TR && t >= nvalid && t < ((nvalid + 15) & ~15)) {
          uint8_t* slot = smem + L::RING_OFF + (g % L::NSLOT) * L::SLOT;
#pragma unroll
          for (int c = 0; c < L::NCL; ++c)
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4*>(slot + c * L::LAT_CHUNK + t * 128 + u * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
        // test hook: withhold the first tile's P-ready arrival
        if (lane == 0 && !(a.fault == 1 && g == 0)) mbar_arrive(&ctl.p_full[g % NPP]);
        // fold the tile FOLD behind (its factor is the oldest in the history), then push this one
        if (k >= FOLD && ok && !fold(g - FOLD, hist[0])) ok = false;
#pragma unroll
        for (int j = 0; j + 1 < FOLD; ++j)
#pragma unroll
          for (int q = 0; q < HPG; ++q) hist[j][q] = hist[j + 1][q];
#pragma unroll
        for (int q = 0; q < HPG; ++q) hist[FOLD - 1][q] = alpha[q];
        if (k == ntiles - 1) {
          // ------------------------------------------------ end of the piece (every warp of the group meets)
          // fold the tiles still outstanding, oldest first
#pragma unroll
          for (int j = 0; j < FOLD; ++j) {
            const int gj = g - FOLD + 1 + j;
            if (gj >= g0 && ok && !fold(gj, hist[j])) ok = false;
          }
          // softmax sums over the CTA's 128 rows
#pragma unroll
          for (int j = 0; j < HPG; ++j) {
            float v = l_part[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) ctl.wsum[quarter][h0 + j] = v;
          }
          if (grp_any(grp, !ok)) { ok = false; break; }
          float inv_l[HPG];
#pragma unroll
          for (int j = 0; j < HPG; ++j) {
            const int hh = h0 + j;
            const float l = (ctl.wsum[0][hh] + ctl.wsum[1][hh]) + (ctl.wsum[2][hh] + ctl.wsum[3][hh]);
            inv_l[j] = l > 0.f ? 1.f / l : 0.f;
            if (t == j && hh < n_h) {
              const float lse = l > 0.f ? (m_ref[j] + log2f(l)) * kLn2 : -INFINITY;
              if (whole) a.lse[(size_t)seq * n_h + hh] = lse;
              else a.part_lse[(size_t)(seq + chunk) * n_h + hh] = lse;
            }
          }
          // o_lat[seq, h, c] (bf16) or the partial slot (fp32); lane t owns latent column mb*128 + t
#pragma unroll
          for (int mb = 0; mb < L::NB; ++mb) {
            const int c = mb * 128 + t;
#pragma unroll
            for (int j = 0; j < HPG; ++j) {
              const int hh = h0 + j;
              if (hh >= n_h) break;
              const float o = o_acc[mb][j] * inv_l[j];
              if (whole)
                static_cast<__nv_bfloat16*>(a.o_lat)[((size_t)seq * n_h + hh) * DC + c] = __float2bfloat16_rn(o);
              else
                a.part_o[((size_t)(seq + chunk) * n_h + hh) * DC + c] = o;
            }
          }
          grp_bar(grp);   // the sum tables are read before the next piece rewrites them
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, L::TMEM_COLS);
}

template <int DC, int DR, int NGRP>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t s, bool* inlined) {
  using L = Shape<DC, DR>;
  const int D = DC + DR;
  CUtensorMap map_lat, map_rope, map_qlat, map_qrope;
  // cache latent part: {64 columns, rows, DC/64 chunks}, chunk outermost
  {
    const uint64_t dims[3] = {64, (uint64_t)a.B * a.max_len, (uint64_t)L::NCL};
    const uint64_t strides[2] = {(uint64_t)D * 2, 128};
    const uint32_t box[3] = {64, TR, (uint32_t)L::NCL};
    if (!make_tmap_3d_bf16_sw128(&map_lat, a.cache, dims, strides, box)) return cudaErrorInvalidValue;
  }
  // cache RoPE part: {DR columns, rows} starting at column DC
  const char* cache_rope = static_cast<const char*>(a.cache) + DC * 2;
  if (!make_tmap_2d_bf16(&map_rope, cache_rope, DR, (uint64_t)a.B * a.max_len, (uint64_t)D * 2, DR, TR,
                         DR == 64 ? 128 : 64))
    return cudaErrorInvalidValue;
  // queries: {64 columns, B * n_h rows} boxes of n_h rows for the latent part, {DR, rows} for RoPE
  if (!make_tmap_2d_bf16(&map_qlat, a.q_abs, DC, (uint64_t)a.B * a.n_h, (uint64_t)D * 2, 64, (uint32_t)a.n_h, 128))
    return cudaErrorInvalidValue;
  const char* q_rope = static_cast<const char*>(a.q_abs) + DC * 2;
  if (!make_tmap_2d_bf16(&map_qrope, q_rope, DR, (uint64_t)a.B * a.n_h, (uint64_t)D * 2, DR, (uint32_t)a.n_h,
                         DR == 64 ? 128 : 64))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_narrow_kernel<DC, DR, NGRP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_DYN);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  DecodeArgs k = a;
  k.inline_plan = (a.B + PLAN_EXTRA) * 4 <= L::PLAN_BYTES;
  *inlined = k.inline_plan != 0;
  if (!k.inline_plan) {
    cudaError_t e = launch_decode_plan(a.seqlens, a.B, a.max_len, a.grid_chunks, 64, a.allow_whole, 2 * TR, a.plan,
                                       a.status, s);
    if (e != cudaSuccess) return e;
  }
  LaunchCfg lc(dim3((unsigned)a.grid_chunks), dim3(96 + 128 * NGRP), L::SMEM_DYN, s);
  cudaError_t e = cudaLaunchKernelEx(&lc.cfg, decode_narrow_kernel<DC, DR, NGRP>, map_lat, map_rope, map_qlat,
                                     map_qrope, k);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool decode_narrow_supported(const mla_handle_s* h) {
  const mla_config_t& c = h->cfg;
  return c.dtype == MLA_BF16 && c.n_h >= 1 && c.n_h <= NPAD && c.d_c == 128 && (c.d_r == 32 || c.d_r == 64);
}

int decode_narrow_chunks(const mla_handle_s* h) { return h->num_sms < 1 ? 1 : h->num_sms; }

cudaError_t launch_decode_narrow(const mla_handle_s* h, const DecodeArgs& a, cudaStream_t s, int* launches) {
  if (!decode_narrow_supported(h)) return cudaErrorInvalidValue;
  // one softmax group of four warps per four heads
  const int n_h = h->cfg.n_h;
  bool inl = false;
  cudaError_t e;
  if (h->cfg.d_r == 32)
    e = n_h <= 4 ? launch_typed<128, 32, 1>(a, s, &inl) : n_h <= 8 ? launch_typed<128, 32, 2>(a, s, &inl)
                                                                   : launch_typed<128, 32, 4>(a, s, &inl);
  else
    e = n_h <= 4 ? launch_typed<128, 64, 1>(a, s, &inl) : n_h <= 8 ? launch_typed<128, 64, 2>(a, s, &inl)
                                                                   : launch_typed<128, 64, 4>(a, s, &inl);
  if (e != cudaSuccess) return e;
  e = launch_decode_combine(a, MLA_BF16, s);
  if (launches) *launches = inl ? 2 : 3;
  return e;
}

}  // namespace mla
