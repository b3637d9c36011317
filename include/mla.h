/*
 * mla.h — C ABI of the B300 (sm_103a) library for one decode step of
 * Multi-head Latent Attention (MLA) over a compressed latent KV cache.
 *
 * The step, as the pages define it (page title, then section):
 *   [MLA]      "MLA：潜在表示压缩与解耦 RoPE"
 *   [Latent]   "Latent 压缩"
 *   [MiniMind] "MiniMind 学习笔记 10：Multi-Latent Attention，从 KV Cache 压缩到 MiniMind 改造思路"
 *
 *   S1  mla_append_cache : c_KV = W_DKV h, k_R = RoPE(W_KR h)  ->  cache row [c_KV | k_R]
 *                          ([MLA] §3 and §6; row layout from [MiniMind] §9)
 *   S2  mla_absorb_q     : c_Q = W_DQ h, q_C = W_UQ c_Q, q_R = RoPE(W_QR c_Q),
 *                          q~_i = W_UK_i^T q_C_i  ->  q_abs row [q~_i | q_R_i]
 *                          ([MLA] §3, §4 matrix absorption, §6)
 *   S3  mla_decode_attn  : s_{i,t} = q_abs_i . row_t / sqrt(d_h + d_r), softmax over t,
 *                          o_lat_i = sum_t a_{i,t} c_KV_t, plus log-sum-exp
 *                          ([MLA] §6 two-part score, §7 scale; [Latent] value deferral)
 *   S4/S5 mla_out_proj   : u = sum_i W_O_i W_UV_i o_lat_i   ([MLA] §4, the u_t formula; §7)
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never frees or keeps them. The memory the library allocates itself is
 *     made in mla_create (RoPE table, status word) and freed in mla_destroy,
 *     plus one fixed 8 MiB scratch array in device global memory that backs
 *     mla_decode_attn_noalloc (defined in the library, so every GPU that loads
 *     it holds the array until the process exits).
 *   - Storage dtype of every activation / weight / cache tensor is the handle's
 *     dtype (MLA_BF16: bf16, MLA_F32: fp32). Arithmetic accumulates in fp32.
 *     LSE is always fp32.
 *   - Weights are row-major [out, in] (nn.Linear layout). Head i owns rows
 *     [i*d_h, (i+1)*d_h) of W_UQ, W_UK, W_UV, rows [i*d_r, (i+1)*d_r) of W_QR
 *     and columns [i*d_h, (i+1)*d_h) of W_O.
 *   - Every pointer must be 16-byte aligned and every tensor dense (row-major,
 *     no padding); otherwise the call returns MLA_ERR_INVALID_ARG and launches
 *     nothing.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronises. Host-side argument errors are
 *     returned immediately. Device-side violations (an index or length out of
 *     range) are clamped or skipped and recorded in the handle's status word,
 *     read with mla_get_device_status. No kernel traps.
 *   - RoPE (the pages do not define it): rotate-half pairs (x_j, x_{j+d_r/2})
 *     turned by pos * base^(-2j/d_r); cos/sin table built in fp64 on the host
 *     and rounded once to fp32.
 *   - Results are deterministic for a fixed (batch, seqlens, device SM count).
 *   - The tensor-core kernels are launched with programmatic dependent launch:
 *     each may start while the previous kernel on the stream drains, but it
 *     reads nothing an earlier kernel wrote, and writes nothing, before that
 *     kernel has completed, so stream order holds as for plain launches. The
 *     calls make no allocation and no synchronisation, so a sequence of them
 *     can be captured into a CUDA graph (after one eager call has set the
 *     kernels' launch attributes); the graph keeps the pointers and sizes of
 *     the captured calls.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_ABI_VERSION 1

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,   /* bad pointer, size, alignment or shape            */
  MLA_ERR_UNSUPPORTED = -2,   /* valid shape this build has no kernel for          */
  MLA_ERR_CUDA = -3,          /* a CUDA runtime / driver call failed               */
  MLA_ERR_DEVICE = -4,        /* status word: a kernel met out-of-range input       */
  MLA_ERR_TIMEOUT = -5,       /* status word: a bounded wait inside a kernel expired */
  MLA_ERR_WORKSPACE = -6      /* workspace pointer NULL or smaller than required   */
} mla_status_t;

typedef enum { MLA_F32 = 0, MLA_BF16 = 1 } mla_dtype_t;

/* Bits of the device status word (mla_get_device_status). */
#define MLA_DEV_SEQLEN_RANGE  0x1  /* seqlens[b] < 0 or > max_len: clamped            */
#define MLA_DEV_POS_RANGE     0x2  /* append: tok_pos[n] outside [0, max_len) or
                                      outside the RoPE table: row skipped             */
#define MLA_DEV_SEQ_RANGE     0x4  /* append: tok_seq[n] outside [0, batch): skipped  */
#define MLA_DEV_QPOS_RANGE    0x8  /* absorb: pos[b] outside the RoPE table: clamped  */
#define MLA_DEV_TIMEOUT       0x10 /* a bounded mbarrier wait expired                  */

/* Layer shape. d_h is the per-head content width and also the value width;
   the softmax scale is 1/sqrt(d_h + d_r) ([MLA] §7). */
typedef struct {
  int32_t d;        /* hidden width                                  */
  int32_t n_h;      /* heads                                         */
  int32_t d_h;      /* per-head content / value width                */
  int32_t d_c;      /* KV latent width (cached)                      */
  int32_t d_r;      /* decoupled RoPE width (cached, shared)         */
  int32_t d_cq;     /* query latent width                            */
  int32_t dtype;    /* mla_dtype_t                                   */
  int32_t max_pos;  /* RoPE table covers positions [0, max_pos)      */
  double rope_base; /* RoPE base (10000 in every shipped workload)   */
} mla_config_t;

typedef struct mla_handle_s* mla_handle_t;

/* Create a handle on the CURRENT CUDA device: validates the shape, builds the
   RoPE table (fp64 on the host, rounded to fp32) and the status word on the
   device. Returns MLA_ERR_INVALID_ARG for non-positive dims, odd d_r, or
   d_c/d_r not multiples of 8; MLA_ERR_CUDA if an allocation fails. */
MLA_API mla_status_t mla_create(const mla_config_t* cfg, mla_handle_t* out);

/* Free what mla_create allocated. Synchronises the device first. */
MLA_API mla_status_t mla_destroy(mla_handle_t handle);

/* Static description of a status code. Never NULL. */
MLA_API const char* mla_status_string(int32_t status);

MLA_API int32_t mla_abi_version(void);

/* S1 — append N tokens to the latent cache ([MLA] §3 c_KV = W_DKV h; §6 k_R =
   RoPE(W_KR h), shared by all heads; row = [c_KV | k_R] per [MiniMind] §9).
     x        [N, d]              hidden states of the tokens
     W_DKV    [d_c, d], W_KR [d_r, d]
     tok_seq  [N] int32 (device)  sequence of token n, in [0, batch)
     tok_pos  [N] int32 (device)  position of token n, in [0, max_len) and < max_pos;
                                  RoPE is applied at this position
     cache    [batch, max_len, d_c + d_r]  row (tok_seq[n], tok_pos[n]) is written;
                                  no other byte of the cache is touched
   N = 0 is a no-op. Out-of-range tok_seq/tok_pos rows are skipped and flagged. */
MLA_API mla_status_t mla_append_cache(mla_handle_t handle, const void* x, int32_t n_tokens,
                              const void* W_DKV, const void* W_KR,
                              const int32_t* tok_seq, const int32_t* tok_pos,
                              void* cache, int32_t batch, int32_t max_len, void* stream);

/* Workspace bytes mla_absorb_q needs for `batch` new tokens (c_Q and q_C). */
MLA_API mla_status_t mla_absorb_q_workspace_size(mla_handle_t handle, int32_t batch, size_t* bytes);

/* S2 — absorbed query of one new token per sequence ([MLA] §3, §4, §6).
     x      [batch, d]
     W_DQ   [d_cq, d], W_UQ [n_h*d_h, d_cq], W_QR [n_h*d_r, d_cq], W_UK [n_h*d_h, d_c]
     pos    [batch] int32 (device)  position of the new token (RoPE of q_R)
     q_abs  [batch, n_h, d_c + d_r] out: [W_UK_i^T q_C_i | RoPE(W_QR_i c_Q)]
     ws     device scratch of at least mla_absorb_q_workspace_size bytes
   c_Q and q_C are stored in the handle's dtype between the projections. */
MLA_API mla_status_t mla_absorb_q(mla_handle_t handle, const void* x, int32_t batch,
                          const void* W_DQ, const void* W_UQ, const void* W_QR, const void* W_UK,
                          const int32_t* pos, void* q_abs, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes mla_decode_attn needs (split plan and split-KV partials). */
MLA_API mla_status_t mla_decode_workspace_size(mla_handle_t handle, int32_t batch, int32_t max_len,
                                       size_t* bytes);

/* S3 — latent-space attention of one query token per sequence over its cache
   rows [0, seqlens[b]) ([MLA] §6 two-part score, §7 softmax scale
   1/sqrt(d_h+d_r); [MiniMind] §12: the query sees every cached row including
   its own; [Latent] value deferral: o_lat_i = sum_t a_{i,t} c_KV_t).
     q_abs    [batch, n_h, d_c + d_r]
     cache    [batch, max_len, d_c + d_r]
     seqlens  [batch] int32 (device) rows to attend, in [0, max_len]; never written.
              Values outside are clamped and flagged (MLA_DEV_SEQLEN_RANGE).
     o_lat    [batch, n_h, d_c] out (handle dtype), normalised by the softmax sum
     lse      [batch, n_h] fp32 out: natural log of sum_t exp(scaled score)
     ws       device scratch of at least mla_decode_workspace_size bytes
   seqlens[b] == 0 gives o_lat = 0 and lse = -inf for that sequence. */
MLA_API mla_status_t mla_decode_attn(mla_handle_t handle, const void* q_abs, const void* cache,
                             int32_t batch, int32_t max_len, const int32_t* seqlens,
                             void* o_lat, float* lse, void* ws, size_t ws_bytes, void* stream);

/* mla_decode_attn without caller workspace and without any allocation. The
   pages have no counterpart to this call: it exists for callers that cannot
   call cudaMalloc — for instance an engine that hands all device memory to its
   own pool at start-up and forbids allocations outside it, or a latency-bound
   loop that cannot afford cudaMalloc's implicit device synchronisation — and
   so cannot create a handle or a workspace.
   Same computation, layouts and results (within rounding) as mla_decode_attn
   on the CUDA-core kernel family; the shape comes as arguments (n_h, d_h, d_c,
   d_r, dtype = mla_dtype_t) instead of a handle.
   Scratch: the split plan and split-KV partials live in one 8 MiB array in
   device global memory, defined in the library; every GPU that loads the
   library holds it until the process exits. Requests whose plan and partials
   do not fit (roughly 4 * n_h * (d_c + 1) * (batch + 1) bytes at the fewest
   splits) return MLA_ERR_WORKSPACE; d_c above 512 returns MLA_ERR_UNSUPPORTED.
   The first call on each device looks up the array's device address (with
   that device current); make that first call before any stream capture. The
   address is kept for the life of the process: after cudaDeviceReset on a
   device, do not call this function on that device again.
   Every call shares the one array, so calls that overlap on the GPU (other
   streams, other host threads on the same device) race and corrupt each
   other's results; serialise them. Out-of-range seqlens are clamped to
   [0, max_len] (their flag is not reported). Asynchronous on `stream`. */
MLA_API mla_status_t mla_decode_attn_noalloc(int32_t n_h, int32_t d_h, int32_t d_c, int32_t d_r, int32_t dtype,
                                     const void* q_abs, const void* cache, int32_t batch, int32_t max_len,
                                     const int32_t* seqlens, void* o_lat, float* lse, void* stream);

/* Workspace bytes mla_out_proj needs (the expanded per-head outputs o). */
MLA_API mla_status_t mla_out_proj_workspace_size(mla_handle_t handle, int32_t batch, size_t* bytes);

/* S4/S5 — u = W_O [W_UV_1 o_lat_1; ...; W_UV_nh o_lat_nh] ([MLA] §4 u_t formula, §7).
     o_lat [batch, n_h, d_c], W_UV [n_h*d_h, d_c], W_O [d, n_h*d_h], u [batch, d] out. */
MLA_API mla_status_t mla_out_proj(mla_handle_t handle, const void* o_lat, int32_t batch,
                          const void* W_UV, const void* W_O, void* u,
                          void* ws, size_t ws_bytes, void* stream);

/* Pre-merged weight forms ([MLA] §4: W^{UQ T} W^{UK} "can be merged ahead of
   time", and the per-head u_t = sum_i W_O_i W_UV_i o_lat_i). Each merge runs
   once per set of weights (a setup step, not part of the decode step); the
   products are accumulated in fp32 and rounded once to the handle's dtype.
   The caller owns every buffer; the calls are asynchronous on `stream`.

   mla_premerge_query_weights: W_QK [n_h, d_c, d_cq] out, W_QK_i = W_UK_i^T W_UQ_i,
     the map that takes c_Q straight to q~_i = W_QK_i c_Q.
     W_UQ [n_h*d_h, d_cq], W_UK [n_h*d_h, d_c] as in mla_absorb_q.
   mla_premerge_output_weights: W_OUV [d, n_h*d_c] out, column block i (columns
     [i*d_c, (i+1)*d_c)) = W_O_i W_UV_i, so that u = W_OUV [o_lat_1; ...; o_lat_nh].
     W_UV [n_h*d_h, d_c], W_O [d, n_h*d_h] as in mla_out_proj.
   Sizes at the DeepSeek-V2 shape: W_QK 201 MB against 92 MB for W_UQ and W_UK,
   W_OUV 671 MB against 185 MB for W_UV and W_O (bf16). */
MLA_API mla_status_t mla_premerge_query_weights(mla_handle_t handle, const void* W_UQ, const void* W_UK,
                                                void* W_QK, void* stream);
MLA_API mla_status_t mla_premerge_output_weights(mla_handle_t handle, const void* W_UV, const void* W_O,
                                                 void* W_OUV, void* stream);

/* S2 with the pre-merged query map: c_Q = W_DQ x, q~_i = W_QK_i c_Q, q_R =
   RoPE(W_QR c_Q), written to q_abs exactly as mla_absorb_q writes it (two
   launches on the tensor-core path: c_Q, then [W_QK ; W_QR] together).
     W_QK from mla_premerge_query_weights; other arguments as in mla_absorb_q;
     ws at least mla_absorb_q_workspace_size bytes (c_Q is kept there). */
MLA_API mla_status_t mla_absorb_q_premerged(mla_handle_t handle, const void* x, int32_t batch,
                                            const void* W_DQ, const void* W_QK, const void* W_QR,
                                            const int32_t* pos, void* q_abs, void* ws, size_t ws_bytes,
                                            void* stream);

/* S4/S5 with the pre-merged output map: u = W_OUV [o_lat_1; ...; o_lat_nh]
   in one launch, without the expanded per-head outputs o (no workspace).
     o_lat [batch, n_h, d_c], W_OUV [d, n_h*d_c], u [batch, d] out. */
MLA_API mla_status_t mla_out_proj_premerged(mla_handle_t handle, const void* o_lat, int32_t batch,
                                            const void* W_OUV, void* u, void* stream);

/* The MHA path for several new tokens per sequence ([Latent]: at prefill MLA
   takes the MHA path, K and V restored from the latent; [MiniMind] §10 naive
   version; §12 causal visibility with a cache). Append the new tokens with
   mla_append_cache first; then:

   mla_project_q: q [n_tokens, n_h, d_h + d_r] = [W_UQ_i c_Q ; RoPE(W_QR_i c_Q)],
     c_Q = W_DQ x, RoPE at pos[n] (device int32 [n_tokens], < max_pos).
     ws: at least mla_absorb_q_workspace_size(handle, n_tokens) bytes.
   mla_materialise_kv: k_c and v_c [n_rows, n_h, d_h] = W_UK_i c_KV and
     W_UV_i c_KV for n_rows cache rows `rows` [n_rows, d_c + d_r] (e.g. the
     whole cache [batch * max_len] rows; rows past a sequence's end produce
     values that no query reads).
   mla_mha_attn: for sequence b and query t < n_q at position q_pos0[b] + t
     (device int32 [batch]; q_pos0[b] + n_q <= max_len, else clamped and
     flagged MLA_DEV_QPOS_RANGE), causal attention over rows 0..q_pos0[b] + t
     with k = [k_c[b, r, i] ; k_R of cache row (b, r)], v = v_c[b, r, i],
     scale 1/sqrt(d_h + d_r).
       q [batch, n_q, n_h, d_h + d_r], k_c / v_c [batch, max_len, n_h, d_h],
       cache [batch, max_len, d_c + d_r] (k_R read from its last d_r columns),
       o [batch, n_q, n_h, d_h] out (normalised), lse [batch, n_q, n_h] fp32 out
       (natural log). d_h <= 128, else MLA_ERR_UNSUPPORTED. The tensor-core
       kernel (V2 head shape) hands out its work items through a device
       counter of the library's, one of 64 that successive launches take in
       turn and leave reset: at most 64 of its launches may be in flight at
       once (across streams), and a captured graph holding one must not be
       replayed on two streams at the same time.
   mla_project_out: u [n_tokens, d] = W_O o for o [n_tokens, n_h * d_h].
   All asynchronous on `stream`; the caller owns every buffer. */
MLA_API mla_status_t mla_project_q(mla_handle_t handle, const void* x, int32_t n_tokens, const void* W_DQ,
                                   const void* W_UQ, const void* W_QR, const int32_t* pos, void* q, void* ws,
                                   size_t ws_bytes, void* stream);
MLA_API mla_status_t mla_materialise_kv(mla_handle_t handle, const void* rows, int32_t n_rows, const void* W_UK,
                                        const void* W_UV, void* k_c, void* v_c, void* stream);
MLA_API mla_status_t mla_mha_attn(mla_handle_t handle, const void* q, int32_t batch, int32_t n_q, const void* k_c,
                                  const void* v_c, const void* cache, int32_t max_len, const int32_t* q_pos0,
                                  void* o, float* lse, void* stream);
MLA_API mla_status_t mla_project_out(mla_handle_t handle, const void* o, int32_t n_tokens, const void* W_O,
                                     void* u, void* stream);

/* S1..S5 in one call ([MLA] §3-§7; [MiniMind] §9-§12): the new token of
   sequence b (x[b], position pos[b]) is written to cache[b, pos[b], :], the
   absorbed queries are formed, attention covers seqlens[b] rows of sequence b
   (pos[b] + 1 for an ordinary step), and u [batch, d] is written. Weights as
   in the four calls above. The workspace (mla_decode_step_workspace_size)
   holds q_abs, o_lat, lse and the stages' scratch; the call launches the same
   kernels as the four calls in sequence, except that S1 and c_Q = W_DQ x share
   one launch when the tensor-core projection kernel takes both. Errors as for
   the four calls; nothing is launched if an argument is rejected. */
MLA_API mla_status_t mla_decode_step_workspace_size(mla_handle_t handle, int32_t batch, int32_t max_len,
                                                    size_t* bytes);
MLA_API mla_status_t mla_decode_step(mla_handle_t handle, const void* x, int32_t batch, const void* W_DKV,
                                     const void* W_KR, const void* W_DQ, const void* W_UQ, const void* W_QR,
                                     const void* W_UK, const void* W_UV, const void* W_O, const int32_t* pos,
                                     const int32_t* seqlens, void* cache, int32_t max_len, void* u, void* ws,
                                     size_t ws_bytes, void* stream);

/* Synchronise `stream`, return the status-word bits accumulated since the last
   call in *bits, and clear them. Returns MLA_ERR_DEVICE if any bit other than
   MLA_DEV_TIMEOUT was set, MLA_ERR_TIMEOUT if that one was, else MLA_OK. */
MLA_API mla_status_t mla_get_device_status(mla_handle_t handle, void* stream, int32_t* bits);

/* Decode-attention kernel family used by mla_decode_attn. AUTO picks the
   tensor-core (tcgen05) kernel where the shape has one, else the CUDA-core one. */
typedef enum { MLA_DECODE_AUTO = 0, MLA_DECODE_SIMT = 1, MLA_DECODE_TCGEN05 = 2 } mla_decode_path_t;
MLA_API mla_status_t mla_set_decode_path(mla_handle_t handle, int32_t path);
/* The path AUTO resolves to for this handle (MLA_DECODE_SIMT or MLA_DECODE_TCGEN05). */
MLA_API mla_status_t mla_get_decode_path(mla_handle_t handle, int32_t* path);

/* Number of split-KV chunks mla_decode_attn cuts the batch's rows into (CTA
   pairs of the tensor-core kernel, CTA columns of the CUDA-core one); 0 (the
   default) = one per pair of SMs / the CUDA-core kernel's usual grid.
   Results differ between chunk counts only by summation order. The decode
   workspace size grows with the count: query mla_decode_workspace_size after
   setting it. Returns MLA_ERR_INVALID_ARG for a negative count or one above
   65535. */
MLA_API mla_status_t mla_set_decode_chunks(mla_handle_t handle, int32_t chunks);

/* Kernel family of the projections (mla_append_cache, mla_absorb_q,
   mla_out_proj). AUTO picks the tensor-core (tcgen05) kernel for bf16 layers
   whose strides it takes (every width a multiple of 8, d_r dividing 128), else
   the CUDA-core one; fp32 layers always use the CUDA-core kernel. */
typedef enum { MLA_PROJ_AUTO = 0, MLA_PROJ_SIMT = 1, MLA_PROJ_TCGEN05 = 2 } mla_proj_path_t;
MLA_API mla_status_t mla_set_proj_path(mla_handle_t handle, int32_t path);

/* The kv_norm variant of the append ([MiniMind] §9: kv_norm = RMSNorm over the
   kv_lora_rank latent, applied before it is cached): with `weight` non-NULL
   (device [d_c], the handle's dtype, 16-byte aligned, owned by the caller and
   read by every later append), mla_append_cache and mla_decode_step replace
   the latent part of each row they append by c / sqrt(mean(c^2) + eps) *
   weight, computed in fp32 from the stored row (so a bf16 row is rounded
   twice); the RoPE key is not normalised. NULL (the default) turns it off.
   Returns MLA_ERR_INVALID_ARG for a misaligned weight or a negative or
   non-finite eps, MLA_ERR_UNSUPPORTED for d_c above 1024. */
MLA_API mla_status_t mla_set_kv_norm(mla_handle_t handle, const void* weight, float eps);

/* Failure-detection controls. Every wait inside the tensor-core kernels is
   bounded: after `cycles` SM clocks without progress (0 restores the default,
   about 2 s) the kernel stops issuing work, waits for its own copies in flight,
   frees its TMEM, sets MLA_DEV_TIMEOUT in the status word and returns, leaving
   the context usable; mla_get_device_status then returns MLA_ERR_TIMEOUT and the
   call's outputs are void. Returns MLA_ERR_INVALID_ARG for a negative count. */
MLA_API mla_status_t mla_set_wait_limit(mla_handle_t handle, int64_t cycles);
/* Test hook for the path above (no GPU fault involved): mode 1 makes the next
   tensor-core decode-attention calls withhold one internal arrival (a barrier
   that nothing else completes), so that their bounded wait runs out; mode 0
   (the default) turns it off. Returns MLA_ERR_INVALID_ARG for other modes. */
MLA_API mla_status_t mla_set_fault_injection(mla_handle_t handle, int32_t mode);

/* Number of kernel launches the last successful call of each entry point made
   (for launch accounting in benchmarks). */
MLA_API mla_status_t mla_last_launch_count(mla_handle_t handle, int32_t* launches);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H_ */
