// TMA tensor-map construction shared by the tcgen05 kernels' host code.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace sl {

// 2-D map over a row-major matrix: inner extent `cols`, outer `rows`, row
// pitch `pitch_bytes`; box (box_cols x box_rows); out-of-bounds boxes read as
// zero.  Rejects (SL_ERR_INVALID) a base or pitch that is not 16-byte aligned.
sl_status make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                   uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw);

}  // namespace sl
