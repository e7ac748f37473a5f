// Library-internal helpers shared by the translation units of the C ABI.
#pragma once

#include <cuda_runtime.h>

namespace sgemm {

// One-time per-device setup (kernel attributes, SM count, workspace pool) for the current
// device; returns its status and the SM count.
cudaError_t device_setup(int *num_sms);

// The stream-ordered workspace pool of the current device (created by device_setup).
cudaMemPool_t workspace_pool();

}  // namespace sgemm
