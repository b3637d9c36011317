// Host-side creation of TMA tensor maps (cuTensorMapEncodeTiled through the
// runtime's driver entry point, so the library needs no -lcuda). Encoded maps
// are cached by their full parameter set (thread-safe), so calls that repeat
// the same tensors skip the driver's encoding.
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace mla {
// 2-D bf16 tensor [outer][inner] with `row_bytes` between rows; box of
// box_inner x box_outer elements, 128-byte swizzle (box_inner * 2 <= 128).
// Returns false if the driver rejects the map.
bool make_tmap_2d_bf16_sw128(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                             uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
// 2-D bf16 tensor with a chosen swizzle span (32, 64 or 128 bytes; box_inner * 2
// must not exceed it).
bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                       uint32_t box_inner, uint32_t box_outer, int swizzle_bytes);
// The same for fp32 elements (box_inner * 4 <= 128).
bool make_tmap_2d_f32_sw128(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
// 3-D bf16 tensor with extents dims[0] (contiguous), dims[1], dims[2] and byte
// strides strides[0] (between dim-1 steps) and strides[1] (between dim-2
// steps); box box[0] x box[1] x box[2], 128-byte swizzle (box[0] * 2 <= 128).
// Elements outside the extents read as zero. Returns false if the driver
// rejects the map.
bool make_tmap_3d_bf16_sw128(CUtensorMap* map, const void* base, const uint64_t dims[3],
                             const uint64_t strides[2], const uint32_t box[3]);
// 4-D form of the above: byte strides strides[0..2] between steps of dims 1..3.
bool make_tmap_4d_bf16_sw128(CUtensorMap* map, const void* base, const uint64_t dims[4],
                             const uint64_t strides[3], const uint32_t box[4]);
}  // namespace mla
