// pkv_stage.h -- copy kernel for staged step inputs and outputs (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

// bytes from src to dst, both device-accessible (device memory, or pinned host
// memory through its device-side address), as one kernel on `stream`.
cudaError_t launch_stage_copy(void* dst, const void* src, int64_t bytes, int num_sms,
                              cudaStream_t stream);

}  // namespace pkv
