#pragma once
#include <cuda.h>

#include "pg_internal.h"

namespace pg {

// 2-D bf16 tensor map with 128-byte swizzle: `inner` contiguous elements per row, `outer` rows
// `row_stride_bytes` apart; boxes of box_inner (<= 64) x box_outer elements; out-of-range
// elements of a box read as zero.
pg_status make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

// 3-D bf16 tensor map with 128-byte swizzle: dims {d0 (contiguous), d1, d2}, d1 and d2 strides
// in bytes, boxes of box0 (<= 64) x box1 x box2; out-of-range elements read as zero.  A box lands in
// shared memory as box2 x box1 rows of box0 elements.
pg_status make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                            uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                            uint32_t box0, uint32_t box1, uint32_t box2);

// 2-D tensor map without swizzle (fp32 or int32 elements, 4 bytes each): `inner` elements per row,
// `outer` rows `row_stride_bytes` apart, boxes of box_inner x box_outer; out-of-range reads are 0.
pg_status make_tmap_2d_b32(CUtensorMap* map, const void* base, bool is_float, uint64_t inner,
                           uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                           uint32_t box_outer);

}  // namespace pg
