// Tensor-core split-KV latent attention for the many-head latent shape
// (n_h = 128, d_c = 512, d_r = 64, bf16): tcgen05.mma with TMEM accumulators,
// TMA-fed shared-memory tiles, warp-specialised pipeline.
//
// What is computed is the same as the CUDA-core kernel (page "MLA：潜在表示压缩
// 与解耦 RoPE", §6 two-part score and §7 softmax with scale 1/sqrt(d_h + d_r);
// page "Latent 压缩", value deferral): for each head i of each sequence,
//   o_lat_i = sum_t softmax_t(q_abs_i . row_t * scale) c_KV_t  and its LSE.
//
// Layout of the work
//   * A CTA pair (cluster 1x2) owns one chunk of the concatenated token space
//     (same plan as the CUDA-core kernel); CTA r holds heads [64r, 64r+64).
//     Both CTAs stream the same cache tiles, the second read mostly from L2.
//   * Per 64-row tile:  S[64 heads x 64 rows] = Q_r . C^T   (M=64, N=64, K=576)
//                       O^T[512 x 64 heads] += C^T . P^T    (4 x M=128, N=64, K=64)
//     The one shared-memory copy of the tile is the K-major B operand of the
//     first product and the MN-major A operand of the second (rows of 128 B,
//     128-byte swizzle), so the latent is read from HBM once per pair.
//   * TMEM (512 columns): S double buffer at columns [0,128), O^T at [256,512).
//   * Warp 0 issues TMA, warp 1 issues MMAs (one thread) and owns TMEM,
//     warps 2-5 run the online softmax, the O rescale and the epilogue.
//   * Online softmax in base 2 with a lazy reference maximum: the running
//     reference moves (and O^T is rescaled in TMEM) only when a head's maximum
//     rises more than 8 above it, so P stays <= 256 and rescales are rare.
//   * Rows past the end of the piece: scores are masked to -inf and the rows
//     are zeroed in shared memory before the PV product (they may hold
//     anything, including NaN).
// Every mbarrier wait is bounded; on expiry the kernel records
// MLA_DEV_TIMEOUT, stops issuing work, and still releases its TMEM.
#include "decode_tc.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int NH = 128, HC = 64, DC = 512, DR = 64, DD = DC + DR;  // shape this kernel serves
constexpr int TN = 64;                   // rows per tile
constexpr int NCHUNK = DD / 64;          // 9 column chunks of 64 (128 B)
constexpr int CHUNK_BYTES = TN * 128;    // 8 KB: 64 rows x 128 B
constexpr int TILE_BYTES = NCHUNK * CHUNK_BYTES;   // 72 KB
constexpr int Q_BYTES = NCHUNK * HC * 128;         // 72 KB
constexpr int P_BYTES = HC * TN * 2;               // 8 KB
constexpr int NSTAGE = 2;
constexpr int SMEM_DYN = Q_BYTES + NSTAGE * TILE_BYTES + P_BYTES + 1024;
constexpr int NTHREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 0;            // S buffers at 0 and 64
constexpr uint32_t O_COL = 256;          // O^T blocks at 256 + 64*blk
constexpr long long WAIT_CYCLES = 4000000000LL;  // ~2 s at 2 GHz
constexpr float kLn2 = 0.693147180559945309f;
constexpr float RESCALE_THRESHOLD = 8.0f;

struct Ctl {
  uint64_t q_full, q_empty, p_full, pv_done;
  uint64_t kv_full[NSTAGE], kv_empty[NSTAGE], s_full[2];
  uint32_t tmem_base;
  int abort;
  float alpha[HC];
  float l[HC];
};

__device__ __forceinline__ void named_sync_softmax() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool named_any_softmax(bool v) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n barrier.cta.red.or.pred po, 1, 128, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)v)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ int find_seq_tc(const int32_t* __restrict__ cum, int B, int r) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cum[mid] <= r) lo = mid; else hi = mid;
  }
  while (lo < B - 1 && cum[lo + 1] <= r) ++lo;
  return lo;
}

// Iterates the pieces (sequence, row range) of this CTA's chunk.
struct PieceIter {
  const int32_t* cum; int B, start, end, b;
  __device__ void init(const int32_t* c, int B_, int chunk) {
    cum = c; B = B_;
    const int cl = cum[B + 1], total = cum[B + 2];
    start = chunk * cl;
    end = min(start + cl, total);
    b = start < end ? find_seq_tc(cum, B, start) : B;
  }
  // next non-empty piece: returns false when done
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

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Ctl& ctl, int32_t* status) {
  if (ctl.abort) return false;
  if (mbar_wait(bar, parity, WAIT_CYCLES)) return true;
  atomicOr(status, MLA_DEV_TIMEOUT);
  ctl.abort = 1;
  return false;
}

__global__ void __cluster_dims__(1, 2, 1) __launch_bounds__(NTHREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv,
                     const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* kv_s = smem + Q_BYTES;
  uint8_t* p_s = kv_s + NSTAGE * TILE_BYTES;
  __shared__ Ctl ctl;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x, half = blockIdx.y;
  const int B = a.B;

  if (threadIdx.x == 0) {
    mbar_init(&ctl.q_full, 1);
    mbar_init(&ctl.q_empty, 1);
    mbar_init(&ctl.p_full, 1);
    mbar_init(&ctl.pv_done, 1);
    for (int s = 0; s < NSTAGE; ++s) { mbar_init(&ctl.kv_full[s], 1); mbar_init(&ctl.kv_empty[s], 1); }
    mbar_init(&ctl.s_full[0], 1);
    mbar_init(&ctl.s_full[1], 1);
    ctl.abort = 0;
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_kv);
      PieceIter it;
      it.init(a.plan, B, chunk);
      int seq, t0, t1;
      bool whole;
      int piece = 0, g = 0;
      bool ok = true;
      while (ok && it.next(seq, t0, t1, whole)) {
        if (piece > 0) ok = wait_or_abort(&ctl.q_empty, (piece - 1) & 1, ctl, a.status);
        if (!ok) break;
        mbar_arrive_expect_tx(&ctl.q_full, Q_BYTES);
        const int qrow = seq * NH + half * HC;
        for (int c = 0; c < NCHUNK; ++c) tma_load_2d(q_s + c * (HC * 128), &map_q, &ctl.q_full, 64 * c, qrow);
        for (int t = t0; t < t1 && ok; t += TN, ++g) {
          const int s = g % NSTAGE;
          if (g >= NSTAGE) ok = wait_or_abort(&ctl.kv_empty[s], ((g / NSTAGE) - 1) & 1, ctl, a.status);
          if (!ok) break;
          mbar_arrive_expect_tx(&ctl.kv_full[s], TILE_BYTES);
          const int row = seq * a.max_len + t;
          uint8_t* dst = kv_s + s * TILE_BYTES;
          for (int c = 0; c < NCHUNK; ++c) tma_load_2d(dst + c * CHUNK_BYTES, &map_kv, &ctl.kv_full[s], 64 * c, row);
        }
        ++piece;
      }
      // On abort, let loads already in flight land before the CTA can exit.
      if (!ok) {
        for (int s = 0; s < NSTAGE; ++s) mbar_wait(&ctl.kv_full[s], 0, WAIT_CYCLES / 4);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16(64, TN, false, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(128, HC, true, false);
      PieceIter it;
      it.init(a.plan, B, chunk);
      // Flatten (piece, tile) so QK of tile g+1 is issued before PV of tile g.
      int seq, t0, t1;
      bool whole;
      int piece = -1, g = 0;
      bool ok = true;
      // state of the tile whose QK has been issued but whose PV has not
      int pend_g = -1;
      bool pend_first = false;
      auto issue_qk = [&](int gg) -> bool {
        const int s = gg % NSTAGE;
        if (!wait_or_abort(&ctl.kv_full[s], (gg / NSTAGE) & 1, ctl, a.status)) return false;
        tc_fence_after();
        const uint32_t qa = smem_u32(q_s), ka = smem_u32(kv_s + s * TILE_BYTES);
        const uint32_t d = tbase + S_COL + (gg & 1) * TN;
#pragma unroll 4
        for (int k = 0; k < DD / 16; ++k) {
          const uint32_t off = (k >> 2) * CHUNK_BYTES + (k & 3) * 32;
          mma_bf16(d, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024), IDESC_QK, k > 0);
        }
        mma_commit(&ctl.s_full[gg & 1]);
        return true;
      };
      auto issue_pv = [&](int gg, bool first_of_piece) -> bool {
        if (!wait_or_abort(&ctl.p_full, gg & 1, ctl, a.status)) return false;
        tc_fence_after();
        const int s = gg % NSTAGE;
        const uint32_t ka = smem_u32(kv_s + s * TILE_BYTES), pa = smem_u32(p_s);
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          const uint32_t d = tbase + O_COL + blk * HC;
#pragma unroll
          for (int k = 0; k < TN / 16; ++k) {
            const uint64_t ad = sdesc_sw128(ka + (2 * blk) * CHUNK_BYTES + k * 16 * 128, CHUNK_BYTES, 1024);
            const uint64_t bd = sdesc_sw128(pa + k * 32, 16, 1024);
            mma_bf16(d, ad, bd, IDESC_PV, (first_of_piece && k == 0) ? 0u : 1u);
          }
        }
        mma_commit(&ctl.kv_empty[s]);
        mma_commit(&ctl.pv_done);
        return true;
      };
      while (ok && it.next(seq, t0, t1, whole)) {
        ++piece;
        if (!wait_or_abort(&ctl.q_full, piece & 1, ctl, a.status)) { ok = false; break; }
        const int ntiles = (t1 - t0 + TN - 1) / TN;
        for (int k = 0; k < ntiles && ok; ++k, ++g) {
          ok = issue_qk(g);
          if (!ok) break;
          if (k == ntiles - 1) mma_commit(&ctl.q_empty);
          if (pend_g >= 0) ok = issue_pv(pend_g, pend_first);
          pend_g = g;
          pend_first = (k == 0);
        }
      }
      if (ok && pend_g >= 0) issue_pv(pend_g, pend_first);
    }
  } else {
    // ------------------------------------------------------------ softmax warps 2..5
    const int quarter = warp & 3;                 // TMEM lane quarter this warp may access
    const int tid = threadIdx.x - 64;             // 0..127
    const bool owner = lane < 16;                 // lanes holding a head row of S (M=64 layout)
    const int h = quarter * 16 + (lane & 15);     // head within this CTA's 64
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = a.scale_log2;
    PieceIter it;
    it.init(a.plan, B, chunk);
    int seq, t0, t1;
    bool whole;
    int g = 0;
    bool ok = true;
    while (ok && it.next(seq, t0, t1, whole)) {
      float m_ref = -INFINITY, l_sum = 0.f;
      const int ntiles = (t1 - t0 + TN - 1) / TN;
      for (int k = 0; k < ntiles; ++k, ++g) {
        const int nvalid = min(TN, t1 - (t0 + k * TN));
        ok = wait_or_abort(&ctl.s_full[g & 1], (g >> 1) & 1, ctl, a.status);
        ok = !named_any_softmax(!ok);  // every softmax thread takes the same branch
        if (!ok) break;
        tc_fence_after();
        float s[TN];
#pragma unroll
        for (int c = 0; c < TN; c += 16) {
          float v[16];
          tmem_ld16(tbase + lane_base + S_COL + (g & 1) * TN + c, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) s[c + i] = v[i];
        }
        tmem_ld_wait();
        float mt = -INFINITY;
#pragma unroll
        for (int i = 0; i < TN; ++i) {
          s[i] = (i < nvalid) ? s[i] * sl2 : -INFINITY;
          mt = fmaxf(mt, s[i]);
        }
        bool need = false;
        float alpha = 1.f;
        if (owner && (m_ref == -INFINITY || mt > m_ref + RESCALE_THRESHOLD)) {
          need = true;
          alpha = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - mt);
          m_ref = mt;
        }
        float psum = 0.f;
        uint32_t packed[TN / 2];
#pragma unroll
        for (int i = 0; i < TN; i += 2) {
          const float p0 = exp2f(s[i] - m_ref), p1 = exp2f(s[i + 1] - m_ref);
          psum += p0 + p1;
          __nv_bfloat162 pr = __floats2bfloat162_rn(p0, p1);
          packed[i / 2] = *reinterpret_cast<uint32_t*>(&pr);
        }
        l_sum = l_sum * alpha + psum;
        if (owner) ctl.alpha[h] = alpha;
        const bool any = named_any_softmax(need && k > 0);
        // PV of the previous tile must be complete: P is single-buffered and O^T may be rescaled.
        if (g > 0) {
          ok = wait_or_abort(&ctl.pv_done, (g - 1) & 1, ctl, a.status);
          ok = !named_any_softmax(!ok);
          if (!ok) break;
          tc_fence_after();
        }
        if (any) {
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
#pragma unroll 1
            for (int c = 0; c < HC; c += 16) {
              float v[16];
              const uint32_t ta = tbase + lane_base + O_COL + blk * HC + c;
              tmem_ld16(ta, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] *= ctl.alpha[c + i];
              tmem_st16(ta, v);
            }
          }
          tmem_st_wait();
        }
        if (nvalid < TN) {
          // zero the tile's rows past the piece end in the 8 latent chunks (PV reads them)
          uint8_t* tile = kv_s + (g % NSTAGE) * TILE_BYTES;
          const int nz = (TN - nvalid) * 8;  // (row, chunk) pairs, 128 B each
          for (int i = tid; i < nz * 8; i += 128) {
            const int pair = i >> 3, part = i & 7;
            const int row = nvalid + pair / 8, c = pair % 8;
            *reinterpret_cast<uint4*>(tile + c * CHUNK_BYTES + row * 128 + part * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        if (owner) {
          // P row h: 64 bf16 = 8 units of 16 B, 128-byte swizzle (unit u at u ^ (h & 7))
          uint8_t* row = p_s + (h >> 3) * 1024 + (h & 7) * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(row + ((u ^ (h & 7)) << 4)) =
                make_uint4(packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_sync_softmax();
        if (tid == 0) mbar_arrive(&ctl.p_full);
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue of this piece
      if (owner) ctl.l[h] = l_sum;
      ok = wait_or_abort(&ctl.pv_done, (g - 1) & 1, ctl, a.status);
      ok = !named_any_softmax(!ok);
      if (!ok) break;
      tc_fence_after();
      const int hg0 = half * HC;
#pragma unroll 1
      for (int blk = 0; blk < 4; ++blk) {
        const int dcol = blk * 128 + quarter * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < HC; c += 16) {
          float v[16];
          tmem_ld16(tbase + lane_base + O_COL + blk * HC + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int hh = c + i;
            const float o = v[i] / ctl.l[hh];
            const long long idx = ((long long)seq * NH + hg0 + hh) * DC + dcol;
            if (whole)
              static_cast<__nv_bfloat16*>(a.o_lat)[idx] = __float2bfloat16_rn(o);
            else
              a.part_o[((long long)(seq + chunk) * NH + hg0 + hh) * DC + dcol] = o;
          }
        }
      }
      if (owner) {
        const float lse = (m_ref + log2f(l_sum)) * kLn2;
        if (whole) a.lse[(long long)seq * NH + hg0 + h] = lse;
        else a.part_lse[(long long)(seq + chunk) * NH + hg0 + h] = lse;
      }
      tc_fence_before();
      named_sync_softmax();
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
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
  CUtensorMap map_q, map_kv;
  if (!make_tmap_2d_bf16_sw128(&map_q, a.q_abs, DD, (uint64_t)a.B * NH, DD * 2, 64, HC))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d_bf16_sw128(&map_kv, a.cache, DD, (uint64_t)a.B * a.max_len, DD * 2, 64, TN))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_decode_plan(a.seqlens, a.B, a.max_len, a.grid_chunks, TN, a.plan, a.status, s);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN);
  if (e != cudaSuccess) return e;
  dim3 grid(a.grid_chunks, 2);
  decode_tc_kernel<<<grid, NTHREADS, SMEM_DYN, s>>>(map_q, map_kv, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_decode_combine(a, MLA_BF16, s);
  if (launches) *launches = 3;
  (void)h;
  return e;
}

}  // namespace mla
