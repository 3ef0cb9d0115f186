// Exhaustive check of bd::f16x2_pow2 (the MXFP4 decode's f16x2 pair of
// powers of two, from one conversion) against bd::f16_pow2 (the same f16
// bits built field by field), for every pair of exponents k in [-300, 0].
// Prints "checked N mismatches M" and exits 0 when the run completed.
#include <cstdio>
#include <cstdint>

#include "bd_device.cuh"

constexpr int kLo = -300, kCount = 301;

__global__ void check(unsigned long long* mismatches) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= kCount * kCount) return;
    const int klo = kLo + i % kCount, khi = kLo + i / kCount;
    const uint32_t want = bd::f16_pow2(klo) | (bd::f16_pow2(khi) << 16);
    if (bd::f16x2_pow2(klo, khi) != want) atomicAdd(mismatches, 1ull);
}

int main() {
    unsigned long long* d = nullptr;
    if (cudaMalloc(&d, sizeof(unsigned long long)) != cudaSuccess) return 1;
    cudaMemset(d, 0, sizeof(unsigned long long));
    const int n = kCount * kCount;
    check<<<(n + 255) / 256, 256>>>(d);
    unsigned long long h = 0;
    if (cudaMemcpy(&h, d, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
    cudaFree(d);
    printf("checked %d mismatches %llu\n", n, h);
    return 0;
}
