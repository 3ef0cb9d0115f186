// Exhaustive check of bd::div6 (the division of a probability block maximum
// by 6) against CUDA's correctly rounded __fdiv_rn(a, 6.0f), bit for bit, and
// of bd::e4m3_div6 (the decode's E4M3 scale byte of a / 6) against
// e4m3(__fdiv_rn(a, 6.0f)), for every binary32 a in [0, 8] (bit patterns
// 0x00000000..0x41000000).  Prints "checked N mismatches M first F scale
// mismatches S first G" and exits 0 when the run completed.
#include <cstdio>
#include <cstdint>

#include "bd_device.cuh"

__global__ void check(unsigned long long n, unsigned long long* mismatches, unsigned int* first) {
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    unsigned long long bad = 0, bad_scale = 0;
    for (unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float a = __uint_as_float((uint32_t)i);
        const float q = __fdiv_rn(a, 6.0f);
        if (__float_as_uint(bd::div6(a)) != __float_as_uint(q)) {
            ++bad;
            atomicMin(&first[0], (unsigned int)i);
        }
        if (bd::e4m3_div6(a) != bd::e4m3(q)) {
            ++bad_scale;
            atomicMin(&first[1], (unsigned int)i);
        }
    }
    if (bad) atomicAdd(&mismatches[0], bad);
    if (bad_scale) atomicAdd(&mismatches[1], bad_scale);
}

int main() {
    const unsigned long long n = 0x41000000ull + 1;   // all patterns up to 8.0f inclusive
    unsigned long long* d_mis = nullptr;
    unsigned int* d_first = nullptr;
    if (cudaMalloc(&d_mis, 2 * sizeof(*d_mis)) != cudaSuccess || cudaMalloc(&d_first, 2 * sizeof(*d_first)) != cudaSuccess) {
        std::printf("cuda allocation failed\n");
        return 2;
    }
    cudaMemset(d_mis, 0, 2 * sizeof(*d_mis));
    cudaMemset(d_first, 0xFF, 2 * sizeof(*d_first));
    check<<<152 * 8, 256>>>(n, d_mis, d_first);
    cudaError_t e = cudaDeviceSynchronize();
    unsigned long long mis[2] = {0, 0};
    unsigned int first[2] = {0, 0};
    cudaMemcpy(mis, d_mis, sizeof(mis), cudaMemcpyDeviceToHost);
    cudaMemcpy(first, d_first, sizeof(first), cudaMemcpyDeviceToHost);
    cudaFree(d_mis);
    cudaFree(d_first);
    if (e != cudaSuccess) {
        std::printf("cuda error %s\n", cudaGetErrorString(e));
        return 2;
    }
    std::printf("checked %llu mismatches %llu first 0x%08x scale mismatches %llu first 0x%08x\n", n, mis[0], first[0],
                mis[1], first[1]);
    return 0;
}
