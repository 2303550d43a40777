// Host-side helpers shared by the launchers (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace fp8act {

// Encode a 2-D uint8 tensor map: `inner` bytes per row (contiguous), `outer`
// rows `row_stride` bytes apart, box of box_inner x box_outer, optionally with
// the 128-byte swizzle. Out-of-bounds boxes read as zero. False on failure.
bool encode_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride,
                       uint32_t box_inner, uint32_t box_outer, bool swizzle128);

}  // namespace fp8act
