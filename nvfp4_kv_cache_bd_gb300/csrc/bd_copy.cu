// Copy between device memory and mapped pinned host memory by a kernel.
//
// On a Grace-Blackwell node the GPU reaches pinned host memory through the
// coherent CPU-GPU link, so a kernel whose threads load and store through the
// host pointer moves the few hundred kilobytes a decode step exchanges with
// the host (its queries in, its outputs out) without a DMA engine's start-up
// cost.  Every SM takes a share of 16-byte words; a tail shorter than 16
// bytes is copied bytewise by the first threads.
#include "bd_copy.h"

#include <algorithm>
#include <cstdint>

namespace bd {
namespace {

__global__ void __launch_bounds__(256) copy_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                                                   size_t bytes) {
    // Programmatic dependent launch: the next kernel in the stream (a decode
    // that streams its static pages first) may start now; this one waits for
    // the preceding grid, which may have written src, before it reads.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t n16 = bytes >> 4;
    const size_t step = (size_t)gridDim.x * blockDim.x;
    const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint4* d = reinterpret_cast<uint4*>(dst);
    const uint4* s = reinterpret_cast<const uint4*>(src);
    for (size_t i = i0; i < n16; i += step) d[i] = s[i];
    const size_t tail = bytes & 15;
    if (i0 < tail) dst[(n16 << 4) + i0] = src[(n16 << 4) + i0];
}

}  // namespace

cudaError_t launch_copy(void* dst, const void* src, size_t bytes, int sms, cudaStream_t s) {
    if (bytes == 0) return cudaSuccess;
    const size_t words = (bytes + 15) >> 4;
    const int blocks = (int)std::min<size_t>((size_t)std::max(sms, 1), (words + 255) / 256);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, copy_kernel, static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src), bytes);
}

}  // namespace bd
