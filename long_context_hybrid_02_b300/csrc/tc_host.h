// Host helpers of the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ha {

// 2-D bf16 tensor map with 128-byte swizzling: `inner` elements per row (contiguous),
// `outer` rows `row_stride_bytes` apart, boxes of box_inner x box_outer
// (box_inner * 2 <= 128).  Out-of-range box elements read as zero.
cudaError_t make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

}  // namespace ha
