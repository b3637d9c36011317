// Host-side creation of TMA tensor maps (cuTensorMapEncodeTiled through the
// runtime's driver entry point, so the library needs no -lcuda).
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace mla {
// 2-D bf16 tensor [outer][inner] with `row_bytes` between rows; box of
// box_inner x box_outer elements, 128-byte swizzle (box_inner * 2 <= 128).
// Returns false if the driver rejects the map.
bool make_tmap_2d_bf16_sw128(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                             uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
}  // namespace mla
