// mla_decode_attn_noalloc: the CUDA-core split-KV decode attention with its
// scratch (split plan, per-chunk partial outputs and log-sum-exps, status word)
// in a file-scope device array instead of caller-allocated workspace, for
// callers that cannot allocate device memory themselves.
//
// The array is a fixed kNoAllocScratchBytes on every GPU that loads this
// library, held until the process exits. Its device address is looked up once
// per device (cudaGetSymbolAddress, with that device current) on the first
// call made on that device, so that first call should come before any stream
// capture. Every call shares the one array: calls that overlap on the GPU
// (different streams, or different host threads on one device) race on it.
#include <math.h>
#include <mutex>

#include "internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr size_t kStatusBytes = 256;                      // status word, padded
constexpr int kMaxDevices = 64;
constexpr int kHeadsPerCta = 16;                          // the CUDA-core kernel's head group

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
int g_num_sms[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the scratch array (looked up on every call: a device
// reset reloads the module and moves it) and the SM count (cached per device).
mla_status_t device_scratch(int dev, void** addr, int* sms) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_num_sms[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return MLA_ERR_CUDA;
    g_num_sms[dev] = n;
  }
  *addr = p;
  *sms = g_num_sms[dev];
  return MLA_OK;
}

}  // namespace

extern "C" mla_status_t mla_decode_attn_noalloc(int32_t n_h, int32_t d_h, int32_t d_c, int32_t d_r, int32_t dtype,
                                                const void* q_abs, const void* cache, int32_t batch,
                                                int32_t max_len, const int32_t* seqlens, void* o_lat, float* lse,
                                                void* stream) {
  if (n_h <= 0 || d_h <= 0 || d_c <= 0 || d_r <= 0 || batch <= 0 || max_len <= 0) return MLA_ERR_INVALID_ARG;
  if (dtype != MLA_BF16 && dtype != MLA_F32) return MLA_ERR_INVALID_ARG;
  if ((d_c % 8) || (d_r % 8)) return MLA_ERR_INVALID_ARG;
  if (!q_abs || !cache || !seqlens || !o_lat || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_abs) || !aligned16(cache) || !aligned16(seqlens) || !aligned16(o_lat) || !aligned16(lse))
    return MLA_ERR_INVALID_ARG;
  if ((long long)batch * max_len >= (1LL << 31)) return MLA_ERR_INVALID_ARG;
  if (d_c > 512) return MLA_ERR_UNSUPPORTED;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  void* base = nullptr;
  int sms = 0;
  const mla_status_t st = device_scratch(dev, &base, &sms);
  if (st != MLA_OK) return st;

  // Chunk count: the CUDA-core kernel's usual grid, reduced until the plan and
  // the partials of (batch + chunks) slots fit the array; too large a batch for
  // even one chunk is rejected.
  const size_t avail = kNoAllocScratchBytes - kStatusBytes;
  const int groups = (n_h + kHeadsPerCta - 1) / kHeadsPerCta;
  int chunks = (4 * sms) / groups;
  if (chunks < 1) chunks = 1;
  while (chunks >= 1 && mla::decode_ws_bytes(batch, n_h, d_c, chunks) > avail) --chunks;
  if (chunks < 1) return MLA_ERR_WORKSPACE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* status = static_cast<int32_t*>(base);
  void* ws = static_cast<unsigned char*>(base) + kStatusBytes;
  // The status word accumulates flags with atomicOr, so it must start at zero.
  // The plan and partials are written in full before they are read.
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return MLA_ERR_CUDA;

  mla::DecodeArgs a{};
  a.q_abs = q_abs; a.cache = cache; a.seqlens = seqlens; a.o_lat = o_lat; a.lse = lse;
  a.B = batch; a.max_len = max_len; a.n_h = n_h; a.d_c = d_c; a.d_r = d_r;
  a.scale_log2 = (float)(1.0 / sqrt((double)(d_h + d_r))) * 1.4426950408889634f;
  a.status = status;
  a.grid_chunks = chunks;
  mla::decode_ws_carve(ws, batch, n_h, d_c, chunks, &a.plan, &a.part_o, &a.part_lse);
  int launches = 0;
  if (mla::launch_decode_simt(a, dtype, s, &launches) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}
