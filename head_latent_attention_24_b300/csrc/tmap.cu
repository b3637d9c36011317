#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <mutex>

#include "tmap.cuh"

namespace mla {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}
// Encoded maps of recent calls, keyed by every encoding parameter: a map is
// a pure function of them (address and layout, no ownership), so a hit is
// always the map the driver would encode again. A decode step encodes about
// twenty maps; the cache keeps that host work off every call after the first.
struct MapKey {
  CUtensorMapDataType dtype;
  uint32_t rank;
  const void* base;
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5];
  CUtensorMapSwizzle swizzle;
  bool operator==(const MapKey& o) const {
    if (dtype != o.dtype || rank != o.rank || base != o.base || swizzle != o.swizzle) return false;
    for (uint32_t i = 0; i < rank; ++i)
      if (dims[i] != o.dims[i] || box[i] != o.box[i]) return false;
    for (uint32_t i = 0; i + 1 < rank; ++i)
      if (strides[i] != o.strides[i]) return false;
    return true;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  uint64_t used;   // 0 = empty
};
constexpr int kMapCache = 128;

bool encode_cached(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                   const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                   CUtensorMapSwizzle swizzle) {
  static std::mutex mu;
  static MapEntry cache[kMapCache];
  static uint64_t clock = 0;
  MapKey key{};
  key.dtype = dtype; key.rank = rank; key.base = base; key.swizzle = swizzle;
  for (uint32_t i = 0; i < rank; ++i) { key.dims[i] = dims[i]; key.box[i] = box[i]; }
  for (uint32_t i = 0; i + 1 < rank; ++i) key.strides[i] = strides[i];
  {
    std::lock_guard<std::mutex> lock(mu);
    for (auto& e : cache)
      if (e.used && e.key == key) {
        e.used = ++clock;
        *map = e.map;
        return true;
      }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, dtype, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(mu);
  MapEntry* victim = &cache[0];
  for (auto& e : cache)
    if (e.used < victim->used) victim = &e;   // an empty slot (0) or the least recently used
  victim->key = key;
  victim->map = *map;
  victim->used = ++clock;
  return true;
}
}  // namespace

bool make_tmap_2d_bf16_sw128(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                             uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  return encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                       uint32_t box_inner, uint32_t box_outer, int swizzle_bytes) {
  CUtensorMapSwizzle sw;
  switch (swizzle_bytes) {
    case 128: sw = CU_TENSOR_MAP_SWIZZLE_128B; break;
    case 64: sw = CU_TENSOR_MAP_SWIZZLE_64B; break;
    case 32: sw = CU_TENSOR_MAP_SWIZZLE_32B; break;
    default: return false;
  }
  if (box_inner * 2 > (uint32_t)swizzle_bytes) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  return encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, sw);
}

bool make_tmap_2d_f32_sw128(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  return encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_tmap_3d_bf16_sw128(CUtensorMap* map, const void* base, const uint64_t dims[3],
                             const uint64_t strides[2], const uint32_t box[3]) {
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides[0], strides[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  return encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, d, st, bx, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_tmap_4d_bf16_sw128(CUtensorMap* map, const void* base, const uint64_t dims[4],
                             const uint64_t strides[3], const uint32_t box[4]) {
  cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
  cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
  return encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, d, st, bx, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace mla
