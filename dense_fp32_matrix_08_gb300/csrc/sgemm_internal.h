// Library-internal helpers shared by the translation units of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace sgemm {

// One-time per-device setup (kernel attributes, SM count, workspace pool) for the current
// device; returns its status and the SM count.
cudaError_t device_setup(int *num_sms);

// The stream-ordered workspace pool of the current device (created by device_setup).
cudaMemPool_t workspace_pool();

// Tensor map (TMA descriptor) of a rows x cols row-major FP32 matrix with row stride ld
// elements (ld * 4 must be a multiple of 16 and ptr 16-byte aligned), box_cols x box_rows
// boxes, optional 128-byte swizzle (box_cols * 4 <= 128 then). Out-of-range elements of a
// box read as zero. Returns false if the driver rejects the description.
bool encode_map_2d(CUtensorMap *map, const float *ptr, long long rows, long long cols,
                   long long ld, int box_cols, int box_rows, bool swizzle128);

}  // namespace sgemm
