// Tensor maps over a paged K or V cache, shared by the attention kernels.
#pragma once

#include <cuda.h>

#include "pa_internal.h"

namespace pa {

// TMA map over a cache [num_blocks][Hkv][16][row_bytes / elem_bytes] with
// 128-byte swizzle.  One box is the 16 rows of one (block, kv head):
// * row_bytes == 256: a single 5-D box (d_lo = 128 bytes, row, d_hi = 2,
//   head, block), landing in shared memory as two 2 KB [row][128 B] halves;
// * row_bytes == 128: a 3-D box (128 bytes, 16 rows of head h at row 16h,
//   block).
// `what` names the caller in error messages.  one_box = false asks for the
// 3-D map with 128-byte boxes on 256-byte rows too (the caller places the
// two halves of a tile itself).
pa_status make_kv_map(CUtensorMap* m, const void* cache, int Hkv, int num_blocks, int row_bytes,
                      int elem_bytes, CUtensorMapDataType dt, const char* what, bool one_box = true);

}  // namespace pa
