// Tensor-core split-KV latent attention for the many-head latent shape
// (n_h = 128, d_c = 512, d_r = 64, bf16): tcgen05.mma with TMEM accumulators,
// TMA-fed shared-memory rings, a CTA pair that splits the work by stage.
//
// What is computed (page "MLA：潜在表示压缩与解耦 RoPE", §6 two-part score and
// §7 softmax with scale 1/sqrt(d_h + d_r); page "Latent 压缩", value deferral):
// for every head i of every sequence
//   s_{i,t} = q_abs_i . row_t * scale,  o_lat_i = sum_t softmax_t(s_{i,t}) c_KV_t,  and the LSE.
//
// Why a pair split by stage. With 128 heads the latent accumulator O
// (128 heads x 512 fp32) fills all 512 TMEM columns of an SM, and the scores
// need columns of their own; the absorbed queries (128 x 576 bf16, 144 KB) do
// not fit next to a pipelined cache tile in shared memory either. So the two
// CTAs of a cluster divide the work:
//   * CTA 0 ("score") holds q~ (the 512 latent columns of q_abs) in TMEM as
//     the A operand and q_R in shared memory, streams full cache tiles
//     (128 rows x 576) through a four-slot ring of 48 KB boxes, and computes
//     S = Q . C^T (M = 128 heads, N = 128 rows, K = 576) into a
//     double-buffered TMEM score block. Eight softmax warps (two per TMEM
//     lane quarter, 64 rows each) turn each score tile into bf16
//     probabilities P and store them, 64 rows at a time, straight from
//     registers into CTA 1's shared memory (st.async, completing on CTA 1's
//     barrier), in the exact layout the MMA reads.
//   * CTA 1 ("value") keeps O = sum_t P_t c_KV_t in all of its TMEM and
//     streams the latent part of the same rows (mostly from L2, where CTA 0's
//     loads left them): O += P . C (M = 128 heads, N = 256 latent columns x 2,
//     K = 64 rows per unit). Its four correction warps apply the rare softmax
//     rescale to O, zero cache rows past a sequence end (P is 0 there, but the
//     rows may hold NaN), and write o_lat / partials at the end of each piece.
// The score SM's copy engine is the scarce resource: it must bring in 1152
// bytes per cached row, close to what one SM's TMA unit moves. So nothing else
// rides on it: P leaves through the threads' asynchronous remote stores,
// not through bulk copies. Only 2 bytes per head and row cross the pair.
// Every MMA has M = 128 and N >= 128, the shapes that run at the full tensor
// rate. One thread issues each CTA's MMAs, and at this rate its instruction
// count matters: the issue loops are unrolled over a tile's boxes and add
// compile-time offsets to shared-memory descriptors built once per kernel.
//
// Softmax: online, in base 2, with a lazy reference maximum per head: the
// reference moves (and O is rescaled) only when a tile's maximum rises more
// than 8 above it, so P <= 256 and rescales are rare after the first tile.
//
// Work split: the plan kernel either gives pair c the whole of sequence c
// (when every sequence has a pair and the longest one costs little more than
// an equal split: no partials, no merge), or lays all sequences' rows end to
// end and cuts them into equal chunks, one per pair; a piece covering a whole
// sequence writes o_lat/lse directly, any other piece a partial slot that the
// LSE combine kernel merges.
//
// Every mbarrier wait is bounded; on expiry a CTA records MLA_DEV_TIMEOUT,
// stops issuing work, waits (bounded) for its own copies in flight, joins the
// final cluster barrier and frees its TMEM.
#include "decode_pair.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int NH = 128, DC = 512, DR = 64, DD = DC + DR;  // the shape this kernel serves
constexpr int TR = 128;                 // cache rows per score tile (MMA N of QK)
constexpr int UR = 64;                  // cache rows per value unit (K of one PV round)
constexpr int NCH = DD / 64;            // 9 column chunks of 64 per row (128 B each)
constexpr int NTHREADS = 320;           // 10 warps
constexpr long long WAIT_CYCLES = 4000000000LL;  // ~2 s
constexpr float kLn2 = 0.693147180559945309f;
constexpr float RESCALE_THRESHOLD = 8.0f;

// Cache tiles are fetched through a 3-D view of the cache, {64 columns, rows,
// 9 column chunks} with the chunk as the outermost dimension, so one TMA box
// brings several 128-byte column chunks of many rows and lands them chunk-major
// ([chunk][row][128 B], 128-byte swizzle): the K-major layout tcgen05 reads.
// CTA 0 shared-memory layout (bytes from the 1024-aligned base)
constexpr int QR_BYTES = NH * 64 * 2;             // 16 KB: q_R of 128 heads
constexpr int S0_CPB = 3;                         // column chunks per score box
constexpr int S0_RING = 4;                        // score ring slots (one box each)
constexpr int S0_CHUNK = TR * 128;                // 16 KB: 128 rows x 64 columns
constexpr int S0_SLOT = S0_CPB * S0_CHUNK;        // 48 KB
constexpr int S0_QR_OFF = 0;
constexpr int S0_RING_OFF = QR_BYTES;
constexpr int S0_END = S0_RING_OFF + S0_RING * S0_SLOT;
// A P unit: P (128 heads x 64 rows bf16, K-major, 128-byte swizzle) followed
// by one 16-byte Info entry per head.
constexpr int NPB = 3;                            // P buffers in CTA 1's shared memory
constexpr int P_BYTES = NH * UR * 2;              // 16 KB
constexpr int P_STRIDE = 18 * 1024;               // P + Info, 1024-aligned
// CTA 1 shared-memory layout
constexpr int S1_CPB = 4;                         // latent chunks per value box
constexpr int S1_RING = 4;
constexpr int S1_CHUNK = UR * 128;                // 8 KB: 64 rows x 64 latent columns
constexpr int S1_SLOT = S1_CPB * S1_CHUNK;        // 32 KB: 64 rows x 256 latent columns
constexpr int S1_P_OFF = 0;
constexpr int S1_RING_OFF = NPB * P_STRIDE;
constexpr int S1_STG_OFF = S1_RING_OFF + S1_RING * S1_SLOT;   // epilogue staging, 16 KB per column half
constexpr int S1_STG = 16 * 1024;
constexpr int S1_END = S1_STG_OFF + 2 * S1_STG;
constexpr int SMEM_DYN = (S0_END > S1_END ? S0_END : S1_END) + 1024;

// TMEM columns
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t QL_COL = 0;          // CTA 0: q~ as the A operand, 256 columns
constexpr uint32_t S_COL = 256;         // CTA 0: two score blocks of 128 columns
// CTA 1: O at columns [0, 512), latent column block nb at nb * 128

constexpr uint32_t FLAG_LAST = 1u;

// Info entry of head h (follows P): x = factor O is rescaled by before this
// unit (1 = none), y = softmax denominator of the piece (if FLAG_LAST),
// z = flags (bit pattern), w unused.
constexpr int P_COPY_BYTES = P_BYTES + NH * 16;
static_assert(P_COPY_BYTES % 16 == 0 && P_COPY_BYTES <= P_STRIDE, "P unit layout");

struct Ctl {
  // CTA 0
  uint64_t r0_full[S0_RING], r0_empty[S0_RING];
  uint64_t q_free, q_ready, s_full[2], s_free[2];
  uint64_t p_free[NPB];       // arrivals: CTA 1's PV MMA commit + CTA 1's Info read
  // CTA 1
  uint64_t r1_full[S1_RING], r1_empty[S1_RING];
  uint64_t p_full[NPB];       // CTA 1's own arming arrival + the remote stores' bytes
  uint64_t unit_ready[NPB];   // CTA 1 correction warps -> MMA
  // PV of the unit in P buffer b complete. One barrier per buffer: a waiter
  // at unit u has seen p_full(u), which implies PV(u - NPB) completed, and
  // PV(u + NPB) needs its unit_ready, so each barrier is within one phase of
  // what its waiter expects (a single barrier could run two phases behind).
  uint64_t pv_done[NPB];
  uint64_t o_free;            // O read out by the 8 epilogue warps
  uint64_t epi_go;            // a piece's last PV is done and inv_l is in shared memory
  uint64_t mma_done;          // every MMA this CTA issued has completed (teardown)
  float inv_l[NH];            // CTA 1: 1 / softmax denominator of the piece being written
  uint32_t tmem_base;
  int abort;
  long long wait_limit;       // cycles before a wait gives up
  float mx[2][2][NH];         // CTA 0: per-half tile maxima, double-buffered by tile
  float lsum[2][NH];          // CTA 0: per-half softmax sums at a piece end
};

__device__ __forceinline__ void sm_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool sm_any(bool v) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n barrier.cta.red.or.pred po, 1, 256, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)v)
      : "memory");
  return out != 0;
}
// The 128 softmax threads of one half (named barriers 3 and 4): all true?
__device__ __forceinline__ bool half_all(int hf, bool v) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n barrier.cta.red.and.pred po, %2, 128, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(3 + hf)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ bool cw_any(bool v) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n barrier.cta.red.or.pred po, 2, 128, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)v)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ int find_seq_p(const int32_t* __restrict__ cum, int B, int r) {
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
    if (cum[B + 3]) {            // whole-sequence plan: chunk c is sequence c
      b = chunk < B ? chunk : B;
      start = chunk < B ? cum[chunk] : 0;
      end = chunk < B ? cum[chunk + 1] : 0;
      return;
    }
    const int cl = cum[B + 1], total = cum[B + 2];
    start = chunk * cl;
    end = min(start + cl, total);
    b = start < end ? find_seq_p(cum, B, start) : B;
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

__device__ __forceinline__ void half_bar(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

// One half (256 columns) of the epilogue of a piece: this thread's head row of
// O, scaled by 1/l, to o_lat (a whole sequence, bf16) or to the piece's fp32
// partial slot. TMEM is read 64 columns at a time; each 128-byte-wide column
// block of the half's 128 rows is written to a swizzled shared staging buffer
// and sent out as one TMA tensor store, so the stores do not queue in the
// threads' load/store path behind the cache stream. The warps release O
// (o_free) after their last TMEM read, before the last stores.
__device__ __forceinline__ void store_o_half(const CUtensorMap* map_ol, const CUtensorMap* map_po, uint32_t taddr,
                                             int half, int row0, int h, bool whole, float inv_l, uint64_t* o_free,
                                             int lane, uint8_t* stg, int bar_id, bool issuer) {
  uint8_t* srow = stg + (h >> 3) * 1024 + (h & 7) * 128;
  const int sw = h & 7;
#pragma unroll 1
  for (int r = 0; r < 4; ++r) {
    float v[64];
    tmem_ld32(taddr + r * 64, v);
    tmem_ld32(taddr + r * 64 + 32, v + 32);
    tmem_ld_wait();
    if (r == 3) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
    }
#pragma unroll
    for (int bx = 0; bx < 2; ++bx) {
      if (whole && bx == 1) break;
      if (issuer) bulk_wait_read<0>();   // the buffer's previous box has been read out
      half_bar(bar_id);
      if (whole) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 pr = __floats2bfloat162_rn(v[8 * u + 2 * e] * inv_l, v[8 * u + 2 * e + 1] * inv_l);
            pk[e] = *reinterpret_cast<uint32_t*>(&pr);
          }
          *reinterpret_cast<uint4*>(srow + ((u ^ sw) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float* x = v + 32 * bx + 4 * u;
          *reinterpret_cast<float4*>(srow + ((u ^ sw) << 4)) =
              make_float4(x[0] * inv_l, x[1] * inv_l, x[2] * inv_l, x[3] * inv_l);
        }
      }
      fence_proxy_async_smem();
      half_bar(bar_id);
      if (issuer) {
        tma_store_2d(whole ? map_ol : map_po, stg, half * 256 + r * 64 + bx * 32, row0);
        bulk_commit();
      }
    }
  }
  if (issuer) bulk_wait_all();   // complete before the buffer is reused or the CTA exits
}

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

__device__ __forceinline__ bool wait_cluster_or_abort(uint64_t* bar, uint32_t parity, Ctl& ctl, int32_t* status) {
  volatile int* ab = reinterpret_cast<volatile int*>(&ctl.abort);
  if (*ab) return false;
  if (mbar_wait_cluster_abortable(bar, parity, ctl.wait_limit, ab)) return true;
  if (!*ab) atomicOr(status, MLA_DEV_TIMEOUT);
  *ab = 1;
  return false;
}

// After an abort: wait (bounded) until every TMA load this producer issued
// into a ring of `ring` slots has landed, so that no copy writes shared memory
// after the CTA has moved on. `issued` loads went to slots 0, 1, 2, ... in
// turn; the last one into slot s filled that slot's phase (last / ring).
__device__ __forceinline__ void drain_ring(uint64_t* full, int ring, int issued) {
  for (int s = 0; s < ring; ++s) {
    if (issued <= s) break;
    const int last = s + ring * ((issued - 1 - s) / ring);
    mbar_wait(&full[s], (uint32_t)((last / ring) & 1), WAIT_CYCLES / 8);
  }
}

__global__ void __launch_bounds__(NTHREADS, 1)
    decode_pair_kernel(const __grid_constant__ CUtensorMap map_kv0, const __grid_constant__ CUtensorMap map_kv1,
                       const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_ol,
                       const __grid_constant__ CUtensorMap map_po, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Ctl ctl;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int chunk = blockIdx.x >> 1;
  const int B = a.B;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S0_RING; ++i) { mbar_init(&ctl.r0_full[i], 1); mbar_init(&ctl.r0_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&ctl.s_full[i], 1); mbar_init(&ctl.s_free[i], 8); }
    mbar_init(&ctl.q_free, 1);
    mbar_init(&ctl.q_ready, 8);
    for (int i = 0; i < S1_RING; ++i) { mbar_init(&ctl.r1_full[i], 1); mbar_init(&ctl.r1_empty[i], 1); }
    for (int i = 0; i < NPB; ++i) {
      mbar_init(&ctl.p_full[i], 1);
      mbar_init(&ctl.p_free[i], 2);
      mbar_init(&ctl.unit_ready[i], 4);
      mbar_init(&ctl.pv_done[i], 1);
    }
    mbar_init(&ctl.o_free, 8);
    mbar_init(&ctl.epi_go, 4);
    mbar_init(&ctl.mma_done, 1);
    ctl.abort = 0;
    ctl.wait_limit = a.wait_cycles > 0 ? a.wait_cycles : WAIT_CYCLES;
    if (cluster_rank() == 1)  // arm the first use of every P buffer
      for (int i = 0; i < NPB; ++i) mbar_arrive_expect_tx(&ctl.p_full[i], P_COPY_BYTES);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tbase = ctl.tmem_base;
  pdl_trigger();
  pdl_wait();      // the plan, the queries and the cache come from earlier kernels
  const uint32_t sbase = smem_u32(smem);
  const float sl2 = a.scale_log2;

  if (rank == 0) {
    // ================================================================ CTA 0: scores and softmax
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) {
        prefetch_tensormap(&map_kv0);
        prefetch_tensormap(&map_q);
        Pieces it;
        it.init(a.plan, B, chunk);
        int seq, t0, t1;
        bool whole;
        int i = 0;
        bool ok = true;
        while (ok && it.next(seq, t0, t1, whole)) {
          // the piece's absorbed queries (128 heads x 576) through the ring, three boxes
          for (int c = 0; c < NCH && ok; c += S0_CPB, ++i) {
            const int sl = i % S0_RING;
            if (i >= S0_RING) ok = wait_or_abort(&ctl.r0_empty[sl], ((i / S0_RING) - 1) & 1, ctl, a.status);
            if (!ok) break;
            mbar_arrive_expect_tx(&ctl.r0_full[sl], S0_SLOT);
            tma_load_3d(smem + S0_RING_OFF + sl * S0_SLOT, &map_q, &ctl.r0_full[sl], 0, seq * NH, c);
          }
          for (int r = t0; r < t1 && ok; r += TR) {
            const int row = seq * a.max_len + r;
            for (int c = 0; c < NCH; c += S0_CPB, ++i) {
              const int sl = i % S0_RING;
              if (i >= S0_RING) ok = wait_or_abort(&ctl.r0_empty[sl], ((i / S0_RING) - 1) & 1, ctl, a.status);
              if (!ok) break;
              mbar_arrive_expect_tx(&ctl.r0_full[sl], S0_SLOT);
              tma_load_3d(smem + S0_RING_OFF + sl * S0_SLOT, &map_kv0, &ctl.r0_full[sl], 0, row, c);
            }
          }
        }
        if (!ok) drain_ring(ctl.r0_full, S0_RING, i);  // no copy lands after the CTA moves on
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer (QK)
      if (lane == 0) {
        constexpr uint32_t IDESC = idesc_bf16(128, TR, false, false);
        Pieces it;
        it.init(a.plan, B, chunk);
        int seq, t0, t1;
        bool whole;
        int piece = 0, g = 0, i = 0;
        bool ok = true;
        const uint64_t ring_desc = sdesc_sw128(sbase + S0_RING_OFF, 16, 1024);
        const uint64_t qr_desc = sdesc_sw128(sbase + S0_QR_OFF, 16, 1024);
        while (ok && it.next(seq, t0, t1, whole)) {
          i += NCH / S0_CPB;   // the query boxes: the softmax warps take them
          ok = wait_or_abort(&ctl.q_ready, piece & 1, ctl, a.status);
          if (!ok) break;
          tc_fence_after();
          for (int r = t0; r < t1 && ok; r += TR, ++g) {
            const int sb = g & 1;
            if (g >= 2) ok = wait_or_abort(&ctl.s_free[sb], ((g >> 1) - 1) & 1, ctl, a.status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d = tbase + S_COL + sb * TR;
#pragma unroll
            for (int bx = 0; bx < NCH / S0_CPB; ++bx, ++i) {
              const int sl = i % S0_RING;
              ok = wait_or_abort(&ctl.r0_full[sl], (i / S0_RING) & 1, ctl, a.status);
              if (!ok) break;
              tc_fence_after();
              const uint64_t bslot = ring_desc + (uint64_t)((sl * S0_SLOT) >> 4);
#pragma unroll
              for (int cc = 0; cc < S0_CPB; ++cc) {
                const int c = bx * S0_CPB + cc;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint64_t bd = bslot + (uint64_t)((cc * S0_CHUNK + k * 32) >> 4);
                  if (c < NCH - 1)
                    mma_bf16_ta(d, tbase + QL_COL + c * 32 + k * 8, bd, IDESC, (c > 0 || k > 0) ? 1u : 0u);
                  else
                    mma_bf16(d, qr_desc + (uint64_t)((k * 32) >> 4), bd, IDESC, 1u);
                }
              }
              mma_commit(&ctl.r0_empty[sl]);
            }
            if (ok) mma_commit(&ctl.s_full[sb]);
          }
          if (ok) mma_commit(&ctl.q_free);
          ++piece;
        }
        // nothing of this CTA's reaches the tensor cores after it moves on
        mma_commit(&ctl.mma_done);
        mbar_wait(&ctl.mma_done, 0, WAIT_CYCLES / 8);
      }
    } else if (warp < 10) {
      // ---------------------------------------------------------- softmax warps 2..9
      const int quarter = warp & 3;
      const int hf = (warp - 2) >> 2;                 // which 64 rows of a tile
      const int h = quarter * 32 + lane;              // head = TMEM lane
      const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
      const uint32_t peer_p = mapa_shared(sbase + S1_P_OFF, 1);
      const uint32_t peer_pfull = mapa_shared(smem_u32(&ctl.p_full[0]), 1);
      Pieces it;
      it.init(a.plan, B, chunk);
      int seq, t0, t1;
      bool whole;
      int piece = 0, g = 0, u = 0, iring = 0;
      bool ok = true;
      while (ok && it.next(seq, t0, t1, whole)) {
        // q~ of this piece's sequence into TMEM (this warp's lanes, its 128 of
        // 256 columns) and q_R into shared memory, from the three ring slots
        // the producer filled with the piece's queries.
        const int len = t1 - t0;
        const int ntiles = (len + TR - 1) / TR;
        const int iq = iring;
        iring += (NCH / S0_CPB) * (1 + ntiles);
        if (piece >= 1) {
          ok = wait_or_abort(&ctl.q_free, (piece - 1) & 1, ctl, a.status);
          ok = !sm_any(!ok);
          if (!ok) break;
          tc_fence_after();
        }
        {
          bool w = true;
          for (int j = 0; j < NCH / S0_CPB; ++j)
            w = w && wait_or_abort(&ctl.r0_full[(iq + j) % S0_RING], ((iq + j) / S0_RING) & 1, ctl, a.status);
          ok = !sm_any(!w);
          if (!ok) break;
          const int roff = (h >> 3) * 1024 + (h & 7) * 128;   // row h of a 128-row chunk (128-byte swizzle)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int c = hf * 4 + jj;
            const uint8_t* rowp = smem + S0_RING_OFF + ((iq + c / S0_CPB) % S0_RING) * S0_SLOT + (c % S0_CPB) * S0_CHUNK + roff;
            uint32_t r[32];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const uint4 x = *reinterpret_cast<const uint4*>(rowp + ((v ^ (h & 7)) << 4));
              r[4 * v] = x.x; r[4 * v + 1] = x.y; r[4 * v + 2] = x.z; r[4 * v + 3] = x.w;
            }
            tmem_st32(tbase + lane_base + QL_COL + hf * 128 + jj * 32, r);
          }
          // q_R: the last chunk, same layout; this half copies 16-byte units 4*hf .. 4*hf+3 of row h
          {
            const uint8_t* src = smem + S0_RING_OFF + ((iq + (NCH - 1) / S0_CPB) % S0_RING) * S0_SLOT +
                                 ((NCH - 1) % S0_CPB) * S0_CHUNK + roff;
            uint8_t* dst = smem + S0_QR_OFF + roff;
#pragma unroll
            for (int v = 4 * hf; v < 4 * hf + 4; ++v) {
              const int o = (v ^ (h & 7)) << 4;
              *reinterpret_cast<uint4*>(dst + o) = *reinterpret_cast<const uint4*>(src + o);
            }
          }
          fence_proxy_async_smem();
          tmem_st_wait();
          tc_fence_before();
          sm_sync();   // every softmax thread is done with the query slots
          if (threadIdx.x == 64)
            for (int j = 0; j < NCH / S0_CPB; ++j) mbar_arrive(&ctl.r0_empty[(iq + j) % S0_RING]);
          __syncwarp();
          // test hook: withhold the first piece's query-ready arrival
          if (lane == 0 && !(a.fault == 1 && piece == 0)) mbar_arrive(&ctl.q_ready);
        }
        float m_ref = -INFINITY, l_part = 0.f;
        for (int k = 0; k < ntiles; ++k, ++g) {
          const int nvalid = min(TR, len - k * TR);
          const bool has_unit = hf == 0 || nvalid > UR;
          const int my_u = u + hf;                     // this half's unit index
          const bool last_tile = k == ntiles - 1;
          const int sb = g & 1;
          const bool w = wait_or_abort(&ctl.s_full[sb], (g >> 1) & 1, ctl, a.status);
          tc_fence_after();
          float s[64];
#pragma unroll
          for (int c = 0; c < 64; c += 16) {
            float v[16];
            tmem_ld16(tbase + lane_base + S_COL + sb * TR + hf * 64 + c, v);
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) s[c + i2] = v[i2];
          }
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.s_free[sb]);
          // scores in base 2, rows past the piece end at -inf; tile maximum
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          if (nvalid == TR) {
#pragma unroll
            for (int i2 = 0; i2 < 64; ++i2) {
              s[i2] *= sl2;
              m4[i2 & 3] = fmaxf(m4[i2 & 3], s[i2]);
            }
          } else {
            const int nv_half = nvalid - hf * 64;
#pragma unroll
            for (int i2 = 0; i2 < 64; ++i2) {
              s[i2] = (i2 < nv_half) ? s[i2] * sl2 : -INFINITY;
              m4[i2 & 3] = fmaxf(m4[i2 & 3], s[i2]);
            }
          }
          ctl.mx[sb][hf][h] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          // one barrier per tile: exchange the halves' maxima and vote on aborting
          if (sm_any(!w || !ok)) { ok = false; break; }
          const float mt = fmaxf(ctl.mx[sb][0][h], ctl.mx[sb][1][h]);
          float alpha = 1.f;
          if (m_ref == -INFINITY || mt > m_ref + RESCALE_THRESHOLD) {
            alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - mt);
            m_ref = mt;
          }
          float p4[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t packed[32];
#pragma unroll
          for (int i2 = 0; i2 < 64; i2 += 2) {
            const float p0 = ex2_approx(s[i2] - m_ref), p1 = ex2_approx(s[i2 + 1] - m_ref);
            p4[(i2 >> 1) & 3] += p0 + p1;
            __nv_bfloat162 pr = __floats2bfloat162_rn(p0, p1);
            packed[i2 / 2] = *reinterpret_cast<uint32_t*>(&pr);
          }
          l_part = l_part * alpha + ((p4[0] + p4[1]) + (p4[2] + p4[3]));
          if (last_tile) {
            ctl.lsum[hf][h] = l_part;
            sm_sync();
          }
          if (has_unit) {
            // the P buffer in CTA 1: its previous unit's PV is done and its Info was read
            const int pb = my_u % NPB;
            bool wf = true;
            if (my_u >= NPB) wf = wait_cluster_or_abort(&ctl.p_free[pb], ((my_u / NPB) - 1) & 1, ctl, a.status);
            if (!half_all(hf, wf)) ok = false;
            if (ok) {
              // P row h of this unit (64 bf16 = 8 chunks of 16 B, 128-byte swizzle) and head h's
              // Info entry, stored into CTA 1's buffer; their bytes complete CTA 1's p_full.
              // Remote stores move twice as fast when each warp store covers whole 128-byte
              // rows, so the 8 lanes of each group first transpose their 8 x 8 chunks
              // (three butterfly stages): lane c of group g then holds chunk c of heads
              // 8g .. 8g+7, and store j writes head 8g+j's row, all 8 chunks across the group.
              const int cg = lane & 7;
#pragma unroll
              for (int st = 4; st >= 1; st >>= 1) {
                const bool up = (cg & st) != 0;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                  if (r & st) continue;
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const uint32_t send = up ? packed[4 * r + e] : packed[4 * (r + st) + e];
                    const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, st);
                    if (up) packed[4 * r + e] = recv; else packed[4 * (r + st) + e] = recv;
                  }
                }
              }
              const uint32_t dst = peer_p + pb * P_STRIDE;
              const uint32_t bar = peer_pfull + pb * 8;
              const int hg = h & ~7;                // this lane's group of 8 heads
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int hh = hg + j;              // the head whose row store j writes
                st_async_v4(dst + (hh >> 3) * 1024 + j * 128 + ((cg ^ j) << 4),
                            make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]), bar);
              }
              const bool last_unit = last_tile && (hf == 1 || nvalid <= UR);
              float l = 0.f;
              if (last_unit) {
                l = ctl.lsum[0][h] + ctl.lsum[1][h];
                const float lse = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
                if (whole) a.lse[(size_t)seq * NH + h] = lse;
                else a.part_lse[(size_t)(seq + chunk) * NH + h] = lse;
              }
              // the rescale applies before the tile's first unit
              st_async_v4(dst + P_BYTES + h * 16,
                          make_uint4(__float_as_uint(hf == 0 ? alpha : 1.f), __float_as_uint(l),
                                     last_unit ? FLAG_LAST : 0u, 0u), bar);
            }
          }
          u += (nvalid > UR) ? 2 : 1;
        }
        if (sm_any(!ok)) break;
        ++piece;
      }
    }
  } else {
    // ================================================================ CTA 1: values
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer (latent part)
      if (lane == 0) {
        prefetch_tensormap(&map_kv1);
        Pieces it;
        it.init(a.plan, B, chunk);
        int seq, t0, t1;
        bool whole;
        int i = 0;
        bool ok = true;
        while (ok && it.next(seq, t0, t1, whole)) {
          for (int r = t0; r < t1 && ok; r += UR) {
            const int row = seq * a.max_len + r;
            for (int j = 0; j < 2; ++j, ++i) {
              const int sl = i % S1_RING;
              if (i >= S1_RING) ok = wait_or_abort(&ctl.r1_empty[sl], ((i / S1_RING) - 1) & 1, ctl, a.status);
              if (!ok) break;
              mbar_arrive_expect_tx(&ctl.r1_full[sl], S1_SLOT);
              tma_load_3d(smem + S1_RING_OFF + sl * S1_SLOT, &map_kv1, &ctl.r1_full[sl], 0, row, j * S1_CPB);
            }
          }
        }
        if (!ok) drain_ring(ctl.r1_full, S1_RING, i);  // no copy lands after the CTA moves on
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer (PV)
      if (lane == 0) {
        constexpr uint32_t IDESC = idesc_bf16(128, 256, false, true);
        const uint64_t p_desc = sdesc_sw128(sbase + S1_P_OFF, 16, 1024);
        const uint64_t v_desc = sdesc_sw128(sbase + S1_RING_OFF, S1_CHUNK, 1024);
        Pieces it;
        it.init(a.plan, B, chunk);
        int seq, t0, t1;
        bool whole;
        int piece = 0, u = 0, i = 0;
        bool ok = true;
        while (ok && it.next(seq, t0, t1, whole)) {
          if (piece > 0) ok = wait_or_abort(&ctl.o_free, (piece - 1) & 1, ctl, a.status);
          bool first = true;
          for (int r = t0; r < t1 && ok; r += UR, ++u) {
            const int pb = u % NPB;
            ok = wait_cluster_or_abort(&ctl.p_full[pb], (u / NPB) & 1, ctl, a.status) &&
                 wait_or_abort(&ctl.unit_ready[pb], (u / NPB) & 1, ctl, a.status);
            if (!ok) break;
            tc_fence_after();
            const uint64_t pd = p_desc + (uint64_t)((pb * P_STRIDE) >> 4);
#pragma unroll
            for (int j = 0; j < 2; ++j, ++i) {
              const int sl = i % S1_RING;
              ok = wait_or_abort(&ctl.r1_full[sl], (i / S1_RING) & 1, ctl, a.status);
              if (!ok) break;
              tc_fence_after();
              // latent columns [256 j, 256 j + 256): four 8 KB chunks, 8 KB apart
              const uint64_t vd = v_desc + (uint64_t)((sl * S1_SLOT) >> 4);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16(tbase + j * 256, pd + (uint64_t)((k * 32) >> 4), vd + (uint64_t)((k * 2048) >> 4), IDESC,
                       (first && k == 0) ? 0u : 1u);
              mma_commit(&ctl.r1_empty[sl]);
            }
            if (!ok) break;
            first = false;
            mma_commit_multicast(&ctl.p_free[pb], 0x1);
            mma_commit(&ctl.pv_done[pb]);
          }
          ++piece;
        }
        // nothing of this CTA's reaches the tensor cores after it moves on
        mma_commit(&ctl.mma_done);
        mbar_wait(&ctl.mma_done, 0, WAIT_CYCLES / 8);
      }
    } else if (warp < 6) {
      // ---------------------------------------------------------- correction / epilogue warps 2..5
      const int quarter = warp & 3;
      const int h = quarter * 32 + lane;
      const int ct = threadIdx.x - 64;   // 0..127
      const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
      const uint32_t peer_pfree = mapa_shared(smem_u32(&ctl.p_free[0]), 0);
      Pieces it;
      it.init(a.plan, B, chunk);
      int seq, t0, t1;
      bool whole;
      int piece = 0, u = 0, i = 0;
      bool ok = true;
      while (ok && it.next(seq, t0, t1, whole)) {
        float inv_l = 0.f;
        bool first = true;
        for (int r = t0; r < t1 && ok; r += UR, ++u, i += 2) {
          const int nrows = min(UR, t1 - r);
          const int pb = u % NPB;
          ok = wait_cluster_or_abort(&ctl.p_full[pb], (u / NPB) & 1, ctl, a.status);
          ok = !cw_any(!ok);
          if (!ok) break;
          const float4 inf = *reinterpret_cast<const float4*>(smem + S1_P_OFF + pb * P_STRIDE + P_BYTES + h * 16);
          const uint32_t flags = __float_as_uint(inf.z);
          const float alpha = inf.x;
          if (flags & FLAG_LAST) {
            const float l = inf.y;
            inv_l = l > 0.f ? 1.f / l : 0.f;
          }
          // Rescale this warp's 32 rows of O when any of them has alpha != 1
          // (never before a piece's first unit: its PV overwrites O).
          if (!first && __any_sync(0xffffffffu, alpha != 1.f)) {
            // O must hold every earlier unit before it is rescaled
            if (!wait_or_abort(&ctl.pv_done[(u - 1) % NPB], ((u - 1) / NPB) & 1, ctl, a.status)) ok = false;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < DC; c += 16) {
              float v[16];
              tmem_ld16(tbase + lane_base + c, v);
              tmem_ld_wait();
#pragma unroll
              for (int i2 = 0; i2 < 16; ++i2) v[i2] *= alpha;
              tmem_st16(tbase + lane_base + c, v);
            }
            tmem_st_wait();
          }
          if (nrows < UR) {
            // zero the unit's rows past the piece end in its 2 slots (8 latent chunks)
            for (int j = 0; j < 2; ++j) {
              const int sl = (i + j) % S1_RING;
              ok = wait_or_abort(&ctl.r1_full[sl], ((i + j) / S1_RING) & 1, ctl, a.status);
              if (!ok) break;
            }
            ok = !cw_any(!ok);
            if (!ok) break;
            const int per_chunk = (UR - nrows) * 8;    // 16-byte words of one chunk's dead rows
            for (int w = ct; w < per_chunk * 8; w += 128) {
              const int ch = w / per_chunk, rem = w % per_chunk;
              const int row = nrows + rem / 8, part = rem % 8;
              uint8_t* base = smem + S1_RING_OFF + ((i + ch / S1_CPB) % S1_RING) * S1_SLOT + (ch % S1_CPB) * S1_CHUNK;
              *reinterpret_cast<uint4*>(base + row * 128 + part * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.unit_ready[pb]);
          ok = !cw_any(!ok);  // also: every correction thread has read this buffer's Info
          if (!ok) break;
          if (ct == 0) {
            mbar_arrive_expect_tx(&ctl.p_full[pb], P_COPY_BYTES);  // arm the buffer's next use
            mbar_arrive_remote(peer_pfree + pb * 8);
          }
          first = false;
          if (flags & FLAG_LAST) {
            // ------------------------------------------------ epilogue of the piece: columns 0..255 here,
            // 256..511 in warps 6..9
            ok = wait_or_abort(&ctl.pv_done[pb], (u / NPB) & 1, ctl, a.status);
            ok = !cw_any(!ok);
            if (!ok) break;
            ctl.inv_l[h] = inv_l;
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.epi_go);
            tc_fence_after();
            store_o_half(&map_ol, &map_po, tbase + lane_base, 0, whole ? seq * NH : (seq + chunk) * NH, h, whole,
                         inv_l, &ctl.o_free, lane, smem + S1_STG_OFF, 2, threadIdx.x == 64);
          }
        }
        ++piece;
      }
    } else if (warp < 10) {
      // ---------------------------------------------------------- epilogue warps 6..9: columns 256..511
      const int quarter = warp & 3;
      const int h = quarter * 32 + lane;
      const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
      Pieces it;
      it.init(a.plan, B, chunk);
      int seq, t0, t1;
      bool whole;
      int piece = 0;
      bool ok = true;
      while (ok && it.next(seq, t0, t1, whole)) {
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl.epi_go, piece & 1, ctl, a.status));
        if (!ok) break;
        const float inv_l = ctl.inv_l[h];
        tc_fence_after();
        store_o_half(&map_ol, &map_po, tbase + lane_base + 256, 1, whole ? seq * NH : (seq + chunk) * NH, h, whole,
                     inv_l, &ctl.o_free, lane, smem + S1_STG_OFF + S1_STG, 3, threadIdx.x == 192);
        ++piece;
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still write into it
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, TMEM_COLS);
}

}  // namespace

bool decode_tc_supported(const mla_handle_s* h) {
  const mla_config_t& c = h->cfg;
  return c.dtype == MLA_BF16 && c.n_h == NH && c.d_c == DC && c.d_r == DR;
}

int decode_tc_chunks(const mla_handle_s* h, int) {
  const int pairs = h->num_sms / 2;
  return pairs < 1 ? 1 : pairs;
}

cudaError_t launch_decode_tc(const mla_handle_s* h, const DecodeArgs& a, cudaStream_t s, int* launches) {
  // Cache viewed as {64 columns, rows, 9 column chunks}: row stride 1152 B,
  // chunk stride 128 B (the chunk is the outer box dimension).
  CUtensorMap map_kv0, map_kv1, map_q, map_ol, map_po;
  const uint64_t dims[3] = {64, (uint64_t)a.B * a.max_len, NCH};
  const uint64_t strides[2] = {DD * 2, 128};
  const uint32_t box0[3] = {64, TR, S0_CPB}, box1[3] = {64, UR, S1_CPB};
  if (!make_tmap_3d_bf16_sw128(&map_kv0, a.cache, dims, strides, box0)) return cudaErrorInvalidValue;
  if (!make_tmap_3d_bf16_sw128(&map_kv1, a.cache, dims, strides, box1)) return cudaErrorInvalidValue;
  // The absorbed queries [B * 128 heads][576] through the same chunk-outer view.
  const uint64_t qdims[3] = {64, (uint64_t)a.B * NH, NCH};
  if (!make_tmap_3d_bf16_sw128(&map_q, a.q_abs, qdims, strides, box0)) return cudaErrorInvalidValue;
  // Epilogue stores: o_lat [B * 128][512] bf16 in 64-column boxes, partials
  // [(B + chunks) * 128][512] fp32 in 32-column boxes, 128 rows each.
  if (!make_tmap_2d_bf16_sw128(&map_ol, a.o_lat, DC, (uint64_t)a.B * NH, DC * 2, 64, NH)) return cudaErrorInvalidValue;
  if (!make_tmap_2d_f32_sw128(&map_po, a.part_o, DC, (uint64_t)(a.B + a.grid_chunks) * NH, DC * 4, 32, NH))
    return cudaErrorInvalidValue;
  // A split costs its pair about a thousand rows of streaming time (the
  // partials' stores, the piece switch and the merge launch).
  constexpr int kSplitCostRows = 1024;
  cudaError_t e = launch_decode_plan(a.seqlens, a.B, a.max_len, a.grid_chunks, UR, a.allow_whole, kSplitCostRows,
                                     a.plan, a.status, s);
  if (e != cudaSuccess) return e;
  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(decode_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  LaunchCfg lc(dim3((unsigned)(2 * a.grid_chunks)), dim3(NTHREADS), SMEM_DYN, s, 2);
  e = cudaLaunchKernelEx(&lc.cfg, decode_pair_kernel, map_kv0, map_kv1, map_q, map_ol, map_po, a);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_decode_combine(a, MLA_BF16, s);
  if (launches) *launches = 3;
  (void)h;
  return e;
}

}  // namespace mla
