// C ABI of the MLA decode library: argument checks, handle state, and the
// launches behind each entry point. See include/mla.h for the contract.
#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <vector>

#include "internal.cuh"
#include "decode_pair.cuh"
#include "decode_narrow.cuh"

using namespace mla;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool on_handle_device(const mla_handle_s* h) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  return dev == h->device;
}

size_t esize(const mla_handle_s* h) { return h->cfg.dtype == MLA_BF16 ? 2 : 4; }

bool use_tc_proj(const mla_handle_s* h, const TcGemm& g) {
  if (h->cfg.dtype != MLA_BF16 || h->proj_path == MLA_PROJ_SIMT) return false;
  return gemm_tc_shape_ok(g);
}

// Segment s of a tensor-core projection: weight rows, output columns and epilogue.
void tc_seg(TcGemm& g, int s, const void* w, int rows, int col0, int epi, void* out, long long ldo,
            long long bo = 0, long long seg_stride = 0, int seg_off = 0) {
  g.w[s] = w; g.rows[s] = rows; g.col0[s] = col0; g.epi[s] = epi; g.out[s] = out; g.ldo[s] = ldo; g.bo[s] = bo;
  g.seg_stride[s] = seg_stride; g.seg_off[s] = seg_off;
  if (s + 1 > g.nseg) g.nseg = s + 1;
}

TcGemm tc_base(const mla_handle_s* h) {
  TcGemm g{};
  g.nseg = 0; g.Z = 1;
  g.rope_cos = h->rope_cos; g.rope_sin = h->rope_sin; g.d_r = h->cfg.d_r; g.max_pos = h->cfg.max_pos;
  g.status = h->status;
  return g;
}

// A tensor-core attention kernel takes this shape: the CTA-pair kernel (128
// heads, d_c 512, d_r 64) or the few-head kernel (n_h <= 16).
bool decode_tc_any(const mla_handle_s* h) { return decode_tc_supported(h) || decode_narrow_supported(h); }

// Split-KV chunk count of the tensor-core family for this shape.
int tc_chunks(const mla_handle_s* h, int batch) {
  return decode_tc_supported(h) ? decode_tc_chunks(h, batch) : decode_narrow_chunks(h);
}

int resolve_decode_path(const mla_handle_s* h) {
  if (h->decode_path == MLA_DECODE_SIMT) return MLA_DECODE_SIMT;
  const bool tc_ok = decode_tc_any(h);
  if (h->decode_path == MLA_DECODE_TCGEN05) return tc_ok ? MLA_DECODE_TCGEN05 : -1;
  return tc_ok ? MLA_DECODE_TCGEN05 : MLA_DECODE_SIMT;
}

// The two tensor-core GEMMs of S4/S5: o_i = W_UV_i o_lat_i batched over the
// heads into `o`, then u = W_O o.
void out_proj_gemms(const mla_handle_s* h, const void* o_lat, int batch, const void* W_UV, const void* W_O,
                    void* u, void* o, TcGemm& g1, TcGemm& g2) {
  const mla_config_t& c = h->cfg;
  g1 = tc_base(h);
  tc_seg(g1, 0, W_UV, c.d_h, 0, EPI_STORE, o, (long long)c.n_h * c.d_h, c.d_h);
  g1.ldw = c.d_c; g1.bw = (long long)c.d_h * c.d_c;
  g1.x = o_lat; g1.ldx = (long long)c.n_h * c.d_c; g1.bx = c.d_c; g1.N = batch; g1.K = c.d_c; g1.Z = c.n_h;
  g2 = tc_base(h);
  tc_seg(g2, 0, W_O, c.d, 0, EPI_STORE, u, c.d);
  g2.ldw = (long long)c.n_h * c.d_h; g2.x = o; g2.ldx = (long long)c.n_h * c.d_h; g2.N = batch;
  g2.K = c.n_h * c.d_h;
}

}  // namespace

extern "C" {

int32_t mla_abi_version(void) { return MLA_ABI_VERSION; }

const char* mla_status_string(int32_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: bad pointer, size, alignment or shape";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: no kernel for this shape";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA call failed";
    case MLA_ERR_DEVICE: return "MLA_ERR_DEVICE: a kernel met out-of-range input (see status bits)";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded wait inside a kernel expired";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing or too small";
    default: return "unknown mla_status_t";
  }
}

mla_status_t mla_create(const mla_config_t* cfg, mla_handle_t* out) {
  if (!cfg || !out) return MLA_ERR_INVALID_ARG;
  *out = nullptr;
  const mla_config_t c = *cfg;
  if (c.d <= 0 || c.n_h <= 0 || c.d_h <= 0 || c.d_c <= 0 || c.d_r <= 0 || c.d_cq <= 0 || c.max_pos <= 0)
    return MLA_ERR_INVALID_ARG;
  if (c.dtype != MLA_BF16 && c.dtype != MLA_F32) return MLA_ERR_INVALID_ARG;
  if ((c.d_r & 1) || (c.d_c % 8) || (c.d_r % 8) || (c.d % 8) || (c.d_cq % 8) || (c.d_h % 8))
    return MLA_ERR_INVALID_ARG;
  if (!(c.rope_base > 1.0) || !isfinite(c.rope_base)) return MLA_ERR_INVALID_ARG;
  if ((long long)c.max_pos * (c.d_r / 2) > (1LL << 31)) return MLA_ERR_INVALID_ARG;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_CUDA;

  mla_handle_s* h = static_cast<mla_handle_s*>(calloc(1, sizeof(mla_handle_s)));
  if (!h) return MLA_ERR_CUDA;
  h->cfg = c;
  h->device = dev;
  h->num_sms = sms;
  h->scale = (float)(1.0 / sqrt((double)(c.d_h + c.d_r)));
  h->decode_path = MLA_DECODE_AUTO;
  h->decode_chunks = 0;

  // RoPE table: angle pos * base^(-2j/d_r) in fp64, cos/sin rounded once to fp32.
  const int half = c.d_r / 2;
  const size_t n = (size_t)c.max_pos * half;
  std::vector<float> cs(n), sn(n);
  std::vector<double> inv(half);
  for (int j = 0; j < half; ++j) inv[j] = pow(c.rope_base, -2.0 * j / c.d_r);
  for (int p = 0; p < c.max_pos; ++p)
    for (int j = 0; j < half; ++j) {
      const double ang = (double)p * inv[j];
      cs[(size_t)p * half + j] = (float)cos(ang);
      sn[(size_t)p * half + j] = (float)sin(ang);
    }
  cudaError_t e = cudaMalloc(&h->rope_cos, n * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&h->rope_sin, n * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&h->status, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemcpy(h->rope_cos, cs.data(), n * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->rope_sin, sn.data(), n * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof(int32_t));
  if (e != cudaSuccess) {
    cudaFree(h->rope_cos);
    cudaFree(h->rope_sin);
    cudaFree(h->status);
    free(h);
    return MLA_ERR_CUDA;
  }
  *out = h;
  return MLA_OK;
}

mla_status_t mla_destroy(mla_handle_t h) {
  if (!h) return MLA_ERR_INVALID_ARG;
  cudaDeviceSynchronize();
  cudaFree(h->rope_cos);
  cudaFree(h->rope_sin);
  cudaFree(h->status);
  free(h);
  return MLA_OK;
}

mla_status_t mla_set_decode_path(mla_handle_t h, int32_t path) {
  if (!h || path < MLA_DECODE_AUTO || path > MLA_DECODE_TCGEN05) return MLA_ERR_INVALID_ARG;
  if (path == MLA_DECODE_TCGEN05 && !decode_tc_any(h)) return MLA_ERR_UNSUPPORTED;
  h->decode_path = path;
  return MLA_OK;
}

mla_status_t mla_set_decode_chunks(mla_handle_t h, int32_t chunks) {
  if (!h || chunks < 0 || chunks > 65535) return MLA_ERR_INVALID_ARG;
  h->decode_chunks = chunks;
  return MLA_OK;
}

mla_status_t mla_get_decode_path(mla_handle_t h, int32_t* path) {
  if (!h || !path) return MLA_ERR_INVALID_ARG;
  *path = resolve_decode_path(h);
  return MLA_OK;
}

mla_status_t mla_set_proj_path(mla_handle_t h, int32_t path) {
  if (!h || path < MLA_PROJ_AUTO || path > MLA_PROJ_TCGEN05) return MLA_ERR_INVALID_ARG;
  if (path == MLA_PROJ_TCGEN05 && h->cfg.dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  h->proj_path = path;
  return MLA_OK;
}

mla_status_t mla_set_kv_norm(mla_handle_t h, const void* weight, float eps) {
  if (!h || (weight && !aligned16(weight)) || !(eps >= 0.f) || !isfinite(eps)) return MLA_ERR_INVALID_ARG;
  if (weight && h->cfg.d_c > 1024) return MLA_ERR_UNSUPPORTED;
  h->kv_norm_weight = weight;
  h->kv_norm_eps = eps;
  return MLA_OK;
}

mla_status_t mla_set_wait_limit(mla_handle_t h, int64_t cycles) {
  if (!h || cycles < 0) return MLA_ERR_INVALID_ARG;
  h->wait_cycles = cycles;
  return MLA_OK;
}

mla_status_t mla_set_fault_injection(mla_handle_t h, int32_t mode) {
  if (!h || mode < 0 || mode > 1) return MLA_ERR_INVALID_ARG;
  h->fault = mode;
  return MLA_OK;
}

mla_status_t mla_last_launch_count(mla_handle_t h, int32_t* launches) {
  if (!h || !launches) return MLA_ERR_INVALID_ARG;
  *launches = h->last_launches;
  return MLA_OK;
}

mla_status_t mla_get_device_status(mla_handle_t h, void* stream, int32_t* bits) {
  if (!h || !bits) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&v, h->status, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof(int32_t));
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  *bits = v;
  if (v & ~MLA_DEV_TIMEOUT) return MLA_ERR_DEVICE;
  if (v & MLA_DEV_TIMEOUT) return MLA_ERR_TIMEOUT;
  return MLA_OK;
}

// ------------------------------------------------------------------- S1
// The kv_norm variant: RMS-normalise the latent of the rows just appended.
static mla_status_t kv_norm_rows(const mla_handle_s* h, void* cache, const int32_t* tok_seq, const int32_t* tok_pos,
                                 int n_tokens, int batch, int max_len, cudaStream_t s, int* launches) {
  if (!h->kv_norm_weight || n_tokens <= 0) return MLA_OK;
  const mla_config_t& c = h->cfg;
  if (launch_kv_norm_rows(cache, h->kv_norm_weight, h->kv_norm_eps, tok_seq, tok_pos, n_tokens, batch, max_len,
                          c.max_pos, c.d_c, c.d_c + c.d_r, c.dtype, s) != cudaSuccess)
    return MLA_ERR_CUDA;
  ++*launches;
  return MLA_OK;
}

// S1 after argument checks; tok_seq == nullptr sends token n to sequence n.
static mla_status_t append_impl(mla_handle_t h, const void* x, int32_t n_tokens, const void* W_DKV, const void* W_KR,
                         const int32_t* tok_seq, const int32_t* tok_pos, void* cache, int32_t batch,
                         int32_t max_len, void* stream) {
  const mla_config_t& c = h->cfg;
  if (c.d_r > 64) return MLA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = c.d_c + c.d_r;
  int launches = 0;
  {
    // One launch: the W_DKV rows then the W_KR rows, scattered to the cache rows.
    TcGemm g = tc_base(h);
    tc_seg(g, 0, W_DKV, c.d_c, 0, EPI_APPEND, cache, 0);
    tc_seg(g, 1, W_KR, c.d_r, c.d_c, EPI_APPEND, cache, 0);
    g.ldw = c.d; g.bw = 0;
    g.x = x; g.ldx = c.d; g.bx = 0; g.K = c.d;
    g.tok_seq = tok_seq; g.tok_pos = tok_pos; g.cache_batch = batch;
    g.max_len = max_len; g.d_c = c.d_c; g.row_width = D;
    g.N = n_tokens;
    if (h->proj_path == MLA_PROJ_TCGEN05 && !use_tc_proj(h, g)) return MLA_ERR_UNSUPPORTED;
    if (use_tc_proj(h, g)) {
      const int chunk = 65535 * 256;
      for (int t0 = 0; t0 < n_tokens; t0 += chunk) {
        TcGemm gc = g;
        gc.N = n_tokens - t0 < chunk ? n_tokens - t0 : chunk;
        gc.x = static_cast<const char*>(x) + (size_t)t0 * c.d * esize(h);
        gc.tok_seq = tok_seq ? tok_seq + t0 : nullptr;
        gc.tok_pos = tok_pos + t0;
        if (launch_gemm_tc(gc, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
        ++launches;
      }
      if (kv_norm_rows(h, cache, tok_seq, tok_pos, n_tokens, batch, max_len, s, &launches) != MLA_OK)
        return MLA_ERR_CUDA;
      h->last_launches = launches;
      return MLA_OK;
    }
  }
  // CUDA-core kernel: two weight blocks, one launch each: c_KV columns then the RoPE columns.
  // The RoPE launch sees both halves of every rotated pair in one tile.
  for (int part = 0; part < 2; ++part) {
    GemmArgs a{};
    a.X = x; a.ldx = c.d; a.bx = 0;
    a.W = part == 0 ? W_DKV : W_KR; a.ldw = c.d; a.bw = 0; a.wlayout = W_NORMAL;
    a.N = n_tokens; a.M = part == 0 ? c.d_c : c.d_r; a.K = c.d; a.batch = 1;
    a.epi = EPI_APPEND;
    a.rope_cos = h->rope_cos; a.rope_sin = h->rope_sin; a.d_r = c.d_r; a.max_pos = c.max_pos;
    a.tok_seq = tok_seq; a.tok_pos = tok_pos; a.cache_batch = batch; a.max_len = max_len;
    a.row_width = D; a.status = h->status;
    // The RoPE block writes at column offset d_c of the row, and every one of
    // its columns is rotated (threshold 0); its d_r <= 64 columns share one tile.
    a.d_c = part == 0 ? c.d_c : 0;
    a.out = part == 0 ? cache : static_cast<char*>(cache) + (size_t)c.d_c * esize(h);
    cudaError_t e;
    // Chunk very long token lists so the grid stays within 65535 rows of tiles.
    const int chunk = 65535 * 64;
    for (int t0 = 0; t0 < n_tokens; t0 += chunk) {
      GemmArgs ac = a;
      ac.N = n_tokens - t0 < chunk ? n_tokens - t0 : chunk;
      ac.X = static_cast<const char*>(x) + (size_t)t0 * c.d * esize(h);
      ac.tok_seq = tok_seq ? tok_seq + t0 : nullptr;
      ac.tok_pos = tok_pos + t0;
      e = launch_gemm_simt(ac, c.dtype, s);
      if (e != cudaSuccess) return MLA_ERR_CUDA;
      ++launches;
    }
  }
  if (kv_norm_rows(h, cache, tok_seq, tok_pos, n_tokens, batch, max_len, s, &launches) != MLA_OK) return MLA_ERR_CUDA;
  h->last_launches = launches;
  return MLA_OK;
}

mla_status_t mla_append_cache(mla_handle_t h, const void* x, int32_t n_tokens, const void* W_DKV,
                              const void* W_KR, const int32_t* tok_seq, const int32_t* tok_pos,
                              void* cache, int32_t batch, int32_t max_len, void* stream) {
  if (!h || n_tokens < 0 || batch <= 0 || max_len <= 0) return MLA_ERR_INVALID_ARG;
  if (n_tokens == 0) { h->last_launches = 0; return MLA_OK; }
  if (!x || !W_DKV || !W_KR || !tok_seq || !tok_pos || !cache) return MLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_DKV) || !aligned16(W_KR) || !aligned16(tok_seq) ||
      !aligned16(tok_pos) || !aligned16(cache))
    return MLA_ERR_INVALID_ARG;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  return append_impl(h, x, n_tokens, W_DKV, W_KR, tok_seq, tok_pos, cache, batch, max_len, stream);
}

// ------------------------------------------------------------------- S2
mla_status_t mla_absorb_q_workspace_size(mla_handle_t h, int32_t batch, size_t* bytes) {
  if (!h || !bytes || batch <= 0) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  *bytes = align_up((size_t)batch * c.d_cq * esize(h), 256) +
           align_up((size_t)batch * c.n_h * c.d_h * esize(h), 256);
  return MLA_OK;
}

mla_status_t mla_absorb_q(mla_handle_t h, const void* x, int32_t batch, const void* W_DQ, const void* W_UQ,
                          const void* W_QR, const void* W_UK, const int32_t* pos, void* q_abs, void* ws,
                          size_t ws_bytes, void* stream) {
  if (!h || batch <= 0 || !x || !W_DQ || !W_UQ || !W_QR || !W_UK || !pos || !q_abs) return MLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_DQ) || !aligned16(W_UQ) || !aligned16(W_QR) || !aligned16(W_UK) ||
      !aligned16(pos) || !aligned16(q_abs) || (ws && !aligned16(ws)))
    return MLA_ERR_INVALID_ARG;
  size_t need = 0;
  mla_absorb_q_workspace_size(h, batch, &need);
  if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  if (64 % c.d_r != 0) return MLA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = c.d_c + c.d_r;
  char* c_q = static_cast<char*>(ws);
  char* q_c = c_q + align_up((size_t)batch * c.d_cq * esize(h), 256);

  {
    TcGemm g1 = tc_base(h);  // c_Q = W_DQ x
    tc_seg(g1, 0, W_DQ, c.d_cq, 0, EPI_STORE, c_q, c.d_cq);
    g1.ldw = c.d; g1.x = x; g1.ldx = c.d; g1.N = batch; g1.K = c.d;
    // q_C = W_UQ c_Q and q_R = RoPE(W_QR c_Q) -> q_abs[b, i, d_c:], one launch (same input)
    TcGemm g2 = tc_base(h);
    tc_seg(g2, 0, W_UQ, c.n_h * c.d_h, 0, EPI_STORE, q_c, (long long)c.n_h * c.d_h);
    tc_seg(g2, 1, W_QR, c.n_h * c.d_r, 0, EPI_ROPE_SEGS, q_abs, (long long)c.n_h * D, 0, D, c.d_c);
    g2.ldw = c.d_cq; g2.x = c_q; g2.ldx = c.d_cq; g2.N = batch; g2.K = c.d_cq; g2.pos = pos;
    TcGemm g4 = tc_base(h);  // q~_i = W_UK_i^T q_C_i -> q_abs[b, i, :d_c]
    tc_seg(g4, 0, W_UK, c.d_c, 0, EPI_STORE, q_abs, (long long)c.n_h * D, D);
    g4.w_transposed = 1; g4.ldw = c.d_c; g4.bw = (long long)c.d_h * c.d_c;
    g4.x = q_c; g4.ldx = (long long)c.n_h * c.d_h; g4.bx = c.d_h; g4.N = batch; g4.K = c.d_h; g4.Z = c.n_h;
    const bool tc = use_tc_proj(h, g1) && use_tc_proj(h, g2) && use_tc_proj(h, g4);
    if (h->proj_path == MLA_PROJ_TCGEN05 && !tc) return MLA_ERR_UNSUPPORTED;
    if (tc) {
      if (launch_gemm_tc(g1, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      if (launch_gemm_tc(g2, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      if (launch_gemm_tc(g4, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      h->last_launches = 3;
      return MLA_OK;
    }
  }
  GemmArgs a{};
  a.batch = 1; a.wlayout = W_NORMAL; a.status = h->status;
  a.rope_cos = h->rope_cos; a.rope_sin = h->rope_sin; a.d_r = c.d_r; a.max_pos = c.max_pos;
  // c_Q = W_DQ x
  a.X = x; a.ldx = c.d; a.W = W_DQ; a.ldw = c.d; a.out = c_q; a.ldo = c.d_cq;
  a.N = batch; a.M = c.d_cq; a.K = c.d; a.epi = EPI_STORE;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  // q_C = W_UQ c_Q
  a.X = c_q; a.ldx = c.d_cq; a.W = W_UQ; a.ldw = c.d_cq; a.out = q_c; a.ldo = (long long)c.n_h * c.d_h;
  a.M = c.n_h * c.d_h; a.K = c.d_cq;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  // q_R = RoPE(W_QR c_Q), written to q_abs[b, i, d_c:]
  a.W = W_QR; a.out = q_abs; a.ldo = (long long)c.n_h * D; a.M = c.n_h * c.d_r;
  a.epi = EPI_ROPE_SEGS; a.pos = pos; a.seg_stride = D; a.seg_off = c.d_c;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  // q~_i = W_UK_i^T q_C_i, batched over heads, written to q_abs[b, i, :d_c]
  GemmArgs t{};
  t.X = q_c; t.ldx = (long long)c.n_h * c.d_h; t.bx = c.d_h;
  t.W = W_UK; t.ldw = c.d_c; t.bw = (long long)c.d_h * c.d_c; t.wlayout = W_TRANSPOSED;
  t.out = q_abs; t.ldo = (long long)c.n_h * D; t.bo = D;
  t.N = batch; t.M = c.d_c; t.K = c.d_h; t.batch = c.n_h; t.epi = EPI_STORE; t.status = h->status;
  if (launch_gemm_simt(t, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  h->last_launches = 4;
  return MLA_OK;
}

// ------------------------------------------------------------------- S3
mla_status_t mla_decode_workspace_size(mla_handle_t h, int32_t batch, int32_t max_len, size_t* bytes) {
  if (!h || !bytes || batch <= 0 || max_len <= 0) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  size_t b = decode_ws_bytes(batch, c.n_h, c.d_c, h->decode_chunks > 0 ? h->decode_chunks : decode_simt_chunks(h));
  if (decode_tc_any(h)) {
    const int ch = h->decode_chunks > 0 ? h->decode_chunks : tc_chunks(h, batch);
    const size_t t = decode_ws_bytes(batch, c.n_h, c.d_c, ch);
    if (t > b) b = t;
  }
  *bytes = b;
  return MLA_OK;
}

mla_status_t mla_decode_attn(mla_handle_t h, const void* q_abs, const void* cache, int32_t batch, int32_t max_len,
                             const int32_t* seqlens, void* o_lat, float* lse, void* ws, size_t ws_bytes,
                             void* stream) {
  if (!h || batch <= 0 || max_len <= 0 || !q_abs || !cache || !seqlens || !o_lat || !lse)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_abs) || !aligned16(cache) || !aligned16(seqlens) || !aligned16(o_lat) || !aligned16(lse) ||
      (ws && !aligned16(ws)))
    return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  if ((long long)batch * max_len >= (1LL << 31)) return MLA_ERR_INVALID_ARG;
  size_t need = 0;
  mla_decode_workspace_size(h, batch, max_len, &need);
  if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const int path = resolve_decode_path(h);
  if (path < 0) return MLA_ERR_UNSUPPORTED;
  if (path == MLA_DECODE_SIMT && c.d_c > 512) return MLA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  DecodeArgs a{};
  a.q_abs = q_abs; a.cache = cache; a.seqlens = seqlens; a.o_lat = o_lat; a.lse = lse;
  a.B = batch; a.max_len = max_len; a.n_h = c.n_h; a.d_c = c.d_c; a.d_r = c.d_r;
  a.scale_log2 = h->scale * 1.4426950408889634f;
  a.status = h->status;
  a.grid_chunks = h->decode_chunks > 0 ? h->decode_chunks
                                        : (path == MLA_DECODE_TCGEN05 ? tc_chunks(h, batch) : decode_simt_chunks(h));
  a.allow_whole = h->decode_chunks == 0;   // a forced chunk count always splits
  a.wait_cycles = h->wait_cycles;
  a.fault = h->fault;
  decode_ws_carve(ws, batch, c.n_h, c.d_c, a.grid_chunks, &a.plan, &a.part_o, &a.part_lse);
  int launches = 0;
  cudaError_t e;
  if (path == MLA_DECODE_TCGEN05)
    e = decode_tc_supported(h) ? launch_decode_tc(h, a, s, &launches) : launch_decode_narrow(h, a, s, &launches);
  else
    e = launch_decode_simt(a, c.dtype, s, &launches);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  h->last_launches = launches;
  return MLA_OK;
}

// ------------------------------------------------------------------- S4/S5
mla_status_t mla_out_proj_workspace_size(mla_handle_t h, int32_t batch, size_t* bytes) {
  if (!h || !bytes || batch <= 0) return MLA_ERR_INVALID_ARG;
  *bytes = align_up((size_t)batch * h->cfg.n_h * h->cfg.d_h * esize(h), 256);
  return MLA_OK;
}

mla_status_t mla_out_proj(mla_handle_t h, const void* o_lat, int32_t batch, const void* W_UV, const void* W_O,
                          void* u, void* ws, size_t ws_bytes, void* stream) {
  if (!h || batch <= 0 || !o_lat || !W_UV || !W_O || !u) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_lat) || !aligned16(W_UV) || !aligned16(W_O) || !aligned16(u) || (ws && !aligned16(ws)))
    return MLA_ERR_INVALID_ARG;
  size_t need = 0;
  mla_out_proj_workspace_size(h, batch, &need);
  if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    TcGemm g1, g2;
    out_proj_gemms(h, o_lat, batch, W_UV, W_O, u, ws, g1, g2);
    const bool tc = use_tc_proj(h, g1) && use_tc_proj(h, g2);
    if (h->proj_path == MLA_PROJ_TCGEN05 && !tc) return MLA_ERR_UNSUPPORTED;
    if (tc) {
      if (launch_gemm_tc(g1, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      if (launch_gemm_tc(g2, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      h->last_launches = 2;
      return MLA_OK;
    }
  }
  // o_i = W_UV_i o_lat_i, batched over heads
  GemmArgs a{};
  a.X = o_lat; a.ldx = (long long)c.n_h * c.d_c; a.bx = c.d_c;
  a.W = W_UV; a.ldw = c.d_c; a.bw = (long long)c.d_h * c.d_c; a.wlayout = W_NORMAL;
  a.out = ws; a.ldo = (long long)c.n_h * c.d_h; a.bo = c.d_h;
  a.N = batch; a.M = c.d_h; a.K = c.d_c; a.batch = c.n_h; a.epi = EPI_STORE; a.status = h->status;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  // u = W_O o
  GemmArgs b{};
  b.X = ws; b.ldx = (long long)c.n_h * c.d_h; b.W = W_O; b.ldw = (long long)c.n_h * c.d_h; b.wlayout = W_NORMAL;
  b.out = u; b.ldo = c.d; b.N = batch; b.M = c.d; b.K = c.n_h * c.d_h; b.batch = 1; b.epi = EPI_STORE;
  b.status = h->status;
  if (launch_gemm_simt(b, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  h->last_launches = 2;
  return MLA_OK;
}

// ------------------------------------------------------------------- pre-merged forms
mla_status_t mla_premerge_query_weights(mla_handle_t h, const void* W_UQ, const void* W_UK, void* W_QK,
                                        void* stream) {
  if (!h || !W_UQ || !W_UK || !W_QK) return MLA_ERR_INVALID_ARG;
  if (!aligned16(W_UQ) || !aligned16(W_UK) || !aligned16(W_QK)) return MLA_ERR_INVALID_ARG;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  if (launch_premerge_query(W_UQ, W_UK, W_QK, c.n_h, c.d_h, c.d_c, c.d_cq, c.dtype,
                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  h->last_launches = 1;
  return MLA_OK;
}

mla_status_t mla_premerge_output_weights(mla_handle_t h, const void* W_UV, const void* W_O, void* W_OUV,
                                         void* stream) {
  if (!h || !W_UV || !W_O || !W_OUV) return MLA_ERR_INVALID_ARG;
  if (!aligned16(W_UV) || !aligned16(W_O) || !aligned16(W_OUV)) return MLA_ERR_INVALID_ARG;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  if (launch_premerge_output(W_UV, W_O, W_OUV, c.n_h, c.d_h, c.d_c, c.d, c.dtype,
                             static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  h->last_launches = 1;
  return MLA_OK;
}

mla_status_t mla_absorb_q_premerged(mla_handle_t h, const void* x, int32_t batch, const void* W_DQ,
                                    const void* W_QK, const void* W_QR, const int32_t* pos, void* q_abs, void* ws,
                                    size_t ws_bytes, void* stream) {
  if (!h || batch <= 0 || !x || !W_DQ || !W_QK || !W_QR || !pos || !q_abs) return MLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_DQ) || !aligned16(W_QK) || !aligned16(W_QR) || !aligned16(pos) ||
      !aligned16(q_abs) || (ws && !aligned16(ws)))
    return MLA_ERR_INVALID_ARG;
  size_t need = 0;
  mla_absorb_q_workspace_size(h, batch, &need);
  if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  if (64 % c.d_r != 0) return MLA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = c.d_c + c.d_r;
  void* c_q = ws;
  {
    TcGemm g1 = tc_base(h);  // c_Q = W_DQ x
    tc_seg(g1, 0, W_DQ, c.d_cq, 0, EPI_STORE, c_q, c.d_cq);
    g1.ldw = c.d; g1.x = x; g1.ldx = c.d; g1.N = batch; g1.K = c.d;
    // [q~ | q_R] = [W_QK ; W_QR] c_Q in one launch: the W_QK rows go to
    // q_abs[b, i, :d_c] in segments of d_c, the W_QR rows get RoPE and go to q_abs[b, i, d_c:]
    TcGemm g2 = tc_base(h);
    tc_seg(g2, 0, W_QK, c.n_h * c.d_c, 0, EPI_SEGS, q_abs, (long long)c.n_h * D, 0, D, 0);
    g2.seg_len[0] = c.d_c;
    tc_seg(g2, 1, W_QR, c.n_h * c.d_r, 0, EPI_ROPE_SEGS, q_abs, (long long)c.n_h * D, 0, D, c.d_c);
    g2.ldw = c.d_cq; g2.x = c_q; g2.ldx = c.d_cq; g2.N = batch; g2.K = c.d_cq; g2.pos = pos;
    const bool tc = use_tc_proj(h, g1) && use_tc_proj(h, g2);
    if (h->proj_path == MLA_PROJ_TCGEN05 && !tc) return MLA_ERR_UNSUPPORTED;
    if (tc) {
      if (launch_gemm_tc(g1, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      if (launch_gemm_tc(g2, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      h->last_launches = 2;
      return MLA_OK;
    }
  }
  GemmArgs a{};
  a.batch = 1; a.wlayout = W_NORMAL; a.status = h->status;
  a.rope_cos = h->rope_cos; a.rope_sin = h->rope_sin; a.d_r = c.d_r; a.max_pos = c.max_pos;
  // c_Q = W_DQ x
  a.X = x; a.ldx = c.d; a.W = W_DQ; a.ldw = c.d; a.out = c_q; a.ldo = c.d_cq;
  a.N = batch; a.M = c.d_cq; a.K = c.d; a.epi = EPI_STORE;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  // q~ = W_QK c_Q into q_abs[b, i, :d_c]
  a.X = c_q; a.ldx = c.d_cq; a.W = W_QK; a.ldw = c.d_cq; a.out = q_abs; a.ldo = (long long)c.n_h * D;
  a.M = c.n_h * c.d_c; a.K = c.d_cq; a.epi = EPI_SEGS; a.seg_len = c.d_c; a.seg_stride = D; a.seg_off = 0;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  // q_R = RoPE(W_QR c_Q) into q_abs[b, i, d_c:]
  a.W = W_QR; a.M = c.n_h * c.d_r; a.epi = EPI_ROPE_SEGS; a.pos = pos; a.seg_stride = D; a.seg_off = c.d_c;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  h->last_launches = 3;
  return MLA_OK;
}

mla_status_t mla_out_proj_premerged(mla_handle_t h, const void* o_lat, int32_t batch, const void* W_OUV, void* u,
                                    void* stream) {
  if (!h || batch <= 0 || !o_lat || !W_OUV || !u) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_lat) || !aligned16(W_OUV) || !aligned16(u)) return MLA_ERR_INVALID_ARG;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int K = c.n_h * c.d_c;
  {
    TcGemm g = tc_base(h);  // u = W_OUV [o_lat_1; ...; o_lat_nh]
    tc_seg(g, 0, W_OUV, c.d, 0, EPI_STORE, u, c.d);
    g.ldw = K; g.x = o_lat; g.ldx = K; g.N = batch; g.K = K;
    const bool tc = use_tc_proj(h, g);
    if (h->proj_path == MLA_PROJ_TCGEN05 && !tc) return MLA_ERR_UNSUPPORTED;
    if (tc) {
      if (launch_gemm_tc(g, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      h->last_launches = 1;
      return MLA_OK;
    }
  }
  GemmArgs a{};
  a.X = o_lat; a.ldx = K; a.W = W_OUV; a.ldw = K; a.wlayout = W_NORMAL; a.out = u; a.ldo = c.d;
  a.N = batch; a.M = c.d; a.K = K; a.batch = 1; a.epi = EPI_STORE; a.status = h->status;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  h->last_launches = 1;
  return MLA_OK;
}

// ------------------------------------------------------------------- the MHA path (several new tokens)
mla_status_t mla_project_q(mla_handle_t h, const void* x, int32_t n_tokens, const void* W_DQ, const void* W_UQ,
                           const void* W_QR, const int32_t* pos, void* q, void* ws, size_t ws_bytes, void* stream) {
  if (!h || n_tokens <= 0 || !x || !W_DQ || !W_UQ || !W_QR || !pos || !q) return MLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_DQ) || !aligned16(W_UQ) || !aligned16(W_QR) || !aligned16(pos) ||
      !aligned16(q) || (ws && !aligned16(ws)))
    return MLA_ERR_INVALID_ARG;
  size_t need = 0;
  mla_absorb_q_workspace_size(h, n_tokens, &need);
  if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  if (64 % c.d_r != 0) return MLA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int DQ = c.d_h + c.d_r;
  void* c_q = ws;
  {
    TcGemm g1 = tc_base(h);  // c_Q = W_DQ x
    tc_seg(g1, 0, W_DQ, c.d_cq, 0, EPI_STORE, c_q, c.d_cq);
    g1.ldw = c.d; g1.x = x; g1.ldx = c.d; g1.N = n_tokens; g1.K = c.d;
    // q = [W_UQ_i c_Q ; RoPE(W_QR_i c_Q)]: segments of d_h and of d_r, one launch
    TcGemm g2 = tc_base(h);
    tc_seg(g2, 0, W_UQ, c.n_h * c.d_h, 0, EPI_SEGS, q, (long long)c.n_h * DQ, 0, DQ, 0);
    g2.seg_len[0] = c.d_h;
    tc_seg(g2, 1, W_QR, c.n_h * c.d_r, 0, EPI_ROPE_SEGS, q, (long long)c.n_h * DQ, 0, DQ, c.d_h);
    g2.ldw = c.d_cq; g2.x = c_q; g2.ldx = c.d_cq; g2.N = n_tokens; g2.K = c.d_cq; g2.pos = pos;
    const bool tc = use_tc_proj(h, g1) && use_tc_proj(h, g2);
    if (h->proj_path == MLA_PROJ_TCGEN05 && !tc) return MLA_ERR_UNSUPPORTED;
    if (tc) {
      if (launch_gemm_tc(g1, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      if (launch_gemm_tc(g2, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      h->last_launches = 2;
      return MLA_OK;
    }
  }
  GemmArgs a{};
  a.batch = 1; a.wlayout = W_NORMAL; a.status = h->status;
  a.rope_cos = h->rope_cos; a.rope_sin = h->rope_sin; a.d_r = c.d_r; a.max_pos = c.max_pos;
  a.X = x; a.ldx = c.d; a.W = W_DQ; a.ldw = c.d; a.out = c_q; a.ldo = c.d_cq;
  a.N = n_tokens; a.M = c.d_cq; a.K = c.d; a.epi = EPI_STORE;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  a.X = c_q; a.ldx = c.d_cq; a.W = W_UQ; a.ldw = c.d_cq; a.out = q; a.ldo = (long long)c.n_h * DQ;
  a.M = c.n_h * c.d_h; a.K = c.d_cq; a.epi = EPI_SEGS; a.seg_len = c.d_h; a.seg_stride = DQ; a.seg_off = 0;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  a.W = W_QR; a.M = c.n_h * c.d_r; a.epi = EPI_ROPE_SEGS; a.pos = pos; a.seg_stride = DQ; a.seg_off = c.d_h;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  h->last_launches = 3;
  return MLA_OK;
}

mla_status_t mla_materialise_kv(mla_handle_t h, const void* rows, int32_t n_rows, const void* W_UK, const void* W_UV,
                                void* k_c, void* v_c, void* stream) {
  if (!h || n_rows <= 0 || !rows || !W_UK || !W_UV || !k_c || !v_c) return MLA_ERR_INVALID_ARG;
  if (!aligned16(rows) || !aligned16(W_UK) || !aligned16(W_UV) || !aligned16(k_c) || !aligned16(v_c))
    return MLA_ERR_INVALID_ARG;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = c.d_c + c.d_r;
  {
    // [k_C | v_C] = [W_UK ; W_UV] c_KV over the rows' latent columns, one launch
    TcGemm g = tc_base(h);
    tc_seg(g, 0, W_UK, c.n_h * c.d_h, 0, EPI_STORE, k_c, (long long)c.n_h * c.d_h);
    tc_seg(g, 1, W_UV, c.n_h * c.d_h, 0, EPI_STORE, v_c, (long long)c.n_h * c.d_h);
    g.ldw = c.d_c; g.x = rows; g.ldx = D; g.N = n_rows; g.K = c.d_c;
    const bool tc = use_tc_proj(h, g);
    if (h->proj_path == MLA_PROJ_TCGEN05 && !tc) return MLA_ERR_UNSUPPORTED;
    if (tc) {
      if (launch_gemm_tc(g, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      h->last_launches = 1;
      return MLA_OK;
    }
  }
  GemmArgs a{};
  a.batch = 1; a.wlayout = W_NORMAL; a.status = h->status; a.epi = EPI_STORE;
  a.X = rows; a.ldx = D; a.W = W_UK; a.ldw = c.d_c; a.out = k_c; a.ldo = (long long)c.n_h * c.d_h;
  a.N = n_rows; a.M = c.n_h * c.d_h; a.K = c.d_c;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  a.W = W_UV; a.out = v_c;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  h->last_launches = 2;
  return MLA_OK;
}

mla_status_t mla_mha_attn(mla_handle_t h, const void* q, int32_t batch, int32_t n_q, const void* k_c,
                          const void* v_c, const void* cache, int32_t max_len, const int32_t* q_pos0, void* o,
                          float* lse, void* stream) {
  if (!h || batch <= 0 || n_q <= 0 || max_len <= 0 || n_q > max_len || !q || !k_c || !v_c || !cache || !q_pos0 ||
      !o || !lse)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_c) || !aligned16(v_c) || !aligned16(cache) || !aligned16(q_pos0) ||
      !aligned16(o) || !aligned16(lse))
    return MLA_ERR_INVALID_ARG;
  if ((long long)batch * max_len >= (1LL << 31)) return MLA_ERR_INVALID_ARG;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  if (c.d_h > 128) return MLA_ERR_UNSUPPORTED;
  MhaArgs a{};
  a.q = q; a.k_c = k_c; a.v_c = v_c; a.cache = cache; a.q_pos0 = q_pos0; a.o = o; a.lse = lse;
  a.B = batch; a.T = n_q; a.max_len = max_len; a.n_h = c.n_h; a.d_h = c.d_h; a.d_c = c.d_c; a.d_r = c.d_r;
  a.scale_log2 = h->scale * 1.4426950408889634f;
  a.wait_cycles = h->wait_cycles;
  a.status = h->status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool tc = h->decode_path != MLA_DECODE_SIMT && mha_tc_supported(h);
  if (h->decode_path == MLA_DECODE_TCGEN05 && !tc) return MLA_ERR_UNSUPPORTED;
  const cudaError_t e = tc ? launch_mha_tc(a, s) : launch_mha_simt(a, c.dtype, s);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  h->last_launches = 1;
  return MLA_OK;
}

mla_status_t mla_project_out(mla_handle_t h, const void* o, int32_t n_tokens, const void* W_O, void* u,
                             void* stream) {
  if (!h || n_tokens <= 0 || !o || !W_O || !u) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(W_O) || !aligned16(u)) return MLA_ERR_INVALID_ARG;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int K = c.n_h * c.d_h;
  {
    TcGemm g = tc_base(h);  // u = W_O o
    tc_seg(g, 0, W_O, c.d, 0, EPI_STORE, u, c.d);
    g.ldw = K; g.x = o; g.ldx = K; g.N = n_tokens; g.K = K;
    const bool tc = use_tc_proj(h, g);
    if (h->proj_path == MLA_PROJ_TCGEN05 && !tc) return MLA_ERR_UNSUPPORTED;
    if (tc) {
      if (launch_gemm_tc(g, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
      h->last_launches = 1;
      return MLA_OK;
    }
  }
  GemmArgs a{};
  a.X = o; a.ldx = K; a.W = W_O; a.ldw = K; a.wlayout = W_NORMAL; a.out = u; a.ldo = c.d;
  a.N = n_tokens; a.M = c.d; a.K = K; a.batch = 1; a.epi = EPI_STORE; a.status = h->status;
  if (launch_gemm_simt(a, c.dtype, s) != cudaSuccess) return MLA_ERR_CUDA;
  h->last_launches = 1;
  return MLA_OK;
}

// ------------------------------------------------------------------- S1..S5
// Workspace of the whole step: q_abs, o_lat and lse, then one region the
// stages use in turn (c_Q and q_C; the split plan and partials; o).
static void step_layout(const mla_handle_s* h, int32_t batch, int32_t max_len, size_t* q_off, size_t* o_off,
                        size_t* l_off, size_t* r_off, size_t* total) {
  const mla_config_t& c = h->cfg;
  size_t off = 0;
  *q_off = off; off += align_up((size_t)batch * c.n_h * (c.d_c + c.d_r) * esize(h), 256);
  *o_off = off; off += align_up((size_t)batch * c.n_h * c.d_c * esize(h), 256);
  *l_off = off; off += align_up((size_t)batch * c.n_h * sizeof(float), 256);
  *r_off = off;
  size_t a = 0, d = 0, o = 0;
  mla_absorb_q_workspace_size(const_cast<mla_handle_t>(h), batch, &a);
  mla_decode_workspace_size(const_cast<mla_handle_t>(h), batch, max_len, &d);
  mla_out_proj_workspace_size(const_cast<mla_handle_t>(h), batch, &o);
  size_t r = a > d ? a : d;
  r = r > o ? r : o;
  *total = off + r;
}

mla_status_t mla_decode_step_workspace_size(mla_handle_t h, int32_t batch, int32_t max_len, size_t* bytes) {
  if (!h || !bytes || batch <= 0 || max_len <= 0) return MLA_ERR_INVALID_ARG;
  size_t q, o, l, r;
  step_layout(h, batch, max_len, &q, &o, &l, &r, bytes);
  return MLA_OK;
}

mla_status_t mla_decode_step(mla_handle_t h, const void* x, int32_t batch, const void* W_DKV, const void* W_KR,
                             const void* W_DQ, const void* W_UQ, const void* W_QR, const void* W_UK,
                             const void* W_UV, const void* W_O, const int32_t* pos, const int32_t* seqlens,
                             void* cache, int32_t max_len, void* u, void* ws, size_t ws_bytes, void* stream) {
  if (!h || batch <= 0 || max_len <= 0) return MLA_ERR_INVALID_ARG;
  if (!x || !W_DKV || !W_KR || !W_DQ || !W_UQ || !W_QR || !W_UK || !W_UV || !W_O || !pos || !seqlens || !cache ||
      !u)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_DKV) || !aligned16(W_KR) || !aligned16(W_DQ) || !aligned16(W_UQ) ||
      !aligned16(W_QR) || !aligned16(W_UK) || !aligned16(W_UV) || !aligned16(W_O) || !aligned16(pos) ||
      !aligned16(seqlens) || !aligned16(cache) || !aligned16(u) || (ws && !aligned16(ws)))
    return MLA_ERR_INVALID_ARG;
  if ((long long)batch * max_len >= (1LL << 31)) return MLA_ERR_INVALID_ARG;
  size_t q_off, o_off, l_off, r_off, need;
  step_layout(h, batch, max_len, &q_off, &o_off, &l_off, &r_off, &need);
  if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
  if (!on_handle_device(h)) return MLA_ERR_INVALID_ARG;
  const mla_config_t& c = h->cfg;
  if (c.d_r > 64 || 64 % c.d_r != 0) return MLA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  void* q_abs = base + q_off;
  void* o_lat = base + o_off;
  float* lse = reinterpret_cast<float*>(base + l_off);
  char* region = base + r_off;
  const size_t region_bytes = ws_bytes - r_off;
  const int D = c.d_c + c.d_r;
  int launches = 0;

  // S1 and c_Q = W_DQ x read the same x: one launch of three weight
  // segments when the tensor-core kernel takes them all (and the rest of S2).
  char* c_q = region;
  char* q_c = c_q + align_up((size_t)batch * c.d_cq * esize(h), 256);
  TcGemm f = tc_base(h);
  tc_seg(f, 0, W_DKV, c.d_c, 0, EPI_APPEND, cache, 0);
  tc_seg(f, 1, W_KR, c.d_r, c.d_c, EPI_APPEND, cache, 0);
  tc_seg(f, 2, W_DQ, c.d_cq, 0, EPI_STORE, c_q, c.d_cq);
  f.ldw = c.d; f.x = x; f.ldx = c.d; f.N = batch; f.K = c.d;
  f.tok_seq = nullptr; f.tok_pos = pos; f.cache_batch = batch; f.max_len = max_len; f.d_c = c.d_c; f.row_width = D;
  TcGemm g2 = tc_base(h);
  tc_seg(g2, 0, W_UQ, c.n_h * c.d_h, 0, EPI_STORE, q_c, (long long)c.n_h * c.d_h);
  tc_seg(g2, 1, W_QR, c.n_h * c.d_r, 0, EPI_ROPE_SEGS, q_abs, (long long)c.n_h * D, 0, D, c.d_c);
  g2.ldw = c.d_cq; g2.x = c_q; g2.ldx = c.d_cq; g2.N = batch; g2.K = c.d_cq; g2.pos = pos;
  TcGemm g4 = tc_base(h);
  tc_seg(g4, 0, W_UK, c.d_c, 0, EPI_STORE, q_abs, (long long)c.n_h * D, D);
  g4.w_transposed = 1; g4.ldw = c.d_c; g4.bw = (long long)c.d_h * c.d_c;
  g4.x = q_c; g4.ldx = (long long)c.n_h * c.d_h; g4.bx = c.d_h; g4.N = batch; g4.K = c.d_h; g4.Z = c.n_h;
  // Every rejection happens here, before the first launch: the decode kernel
  // family, and a forced tensor-core projection path the shapes do not take.
  const int dpath = resolve_decode_path(h);
  if (dpath < 0 || (dpath == MLA_DECODE_SIMT && c.d_c > 512)) return MLA_ERR_UNSUPPORTED;
  const bool tc_front = batch <= 65535 * 256 && use_tc_proj(h, f) && use_tc_proj(h, g2) && use_tc_proj(h, g4);
  TcGemm o1, o2;
  out_proj_gemms(h, o_lat, batch, W_UV, W_O, u, region, o1, o2);
  if (h->proj_path == MLA_PROJ_TCGEN05 && !(tc_front && use_tc_proj(h, o1) && use_tc_proj(h, o2)))
    return MLA_ERR_UNSUPPORTED;
  mla_status_t st;
  if (tc_front) {
    if (launch_gemm_tc(f, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
    if (kv_norm_rows(h, cache, nullptr, pos, batch, batch, max_len, s, &launches) != MLA_OK) return MLA_ERR_CUDA;
    if (launch_gemm_tc(g2, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
    if (launch_gemm_tc(g4, h->num_sms, s) != cudaSuccess) return MLA_ERR_CUDA;
    launches += 3;
  } else {
    st = append_impl(h, x, batch, W_DKV, W_KR, nullptr, pos, cache, batch, max_len, stream);
    if (st != MLA_OK) return st;
    launches += h->last_launches;
    st = mla_absorb_q(h, x, batch, W_DQ, W_UQ, W_QR, W_UK, pos, q_abs, region, region_bytes, stream);
    if (st != MLA_OK) return st;
    launches += h->last_launches;
  }
  st = mla_decode_attn(h, q_abs, cache, batch, max_len, seqlens, o_lat, lse, region, region_bytes, stream);
  if (st != MLA_OK) return st;
  launches += h->last_launches;
  st = mla_out_proj(h, o_lat, batch, W_UV, W_O, u, region, region_bytes, stream);
  if (st != MLA_OK) return st;
  launches += h->last_launches;
  h->last_launches = launches;
  return MLA_OK;
}

}  // extern "C"
