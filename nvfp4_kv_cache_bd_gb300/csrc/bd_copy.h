// Launcher of the host/device copy kernel (bd_copy.cu) behind bd_copy_async.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

namespace bd {

// Copy `bytes` bytes from src to dst (16-byte aligned, not overlapping, each
// device memory or mapped pinned host memory) with at most `sms` CTAs.
cudaError_t launch_copy(void* dst, const void* src, size_t bytes, int sms, cudaStream_t s);

}  // namespace bd
