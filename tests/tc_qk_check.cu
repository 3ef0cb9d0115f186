// Single-page check of the decode's tensor-core QK product: one CTA runs the
// library's own tcgen05 helpers (bd_device.cuh) on one packed K record and
// one token's packed query, laid out exactly as the decode's MMA warp lays
// them out, and writes the 128 x 8 fp32 scores
// S[t][2 hh + term] = Khat_t . Qhat_{4h+hh, term} (block scales applied,
// per-tensor scales not).
//
//   tc_qk_check <in> <out>
//     in : int32 format (0 NVFP4, 1 MXFP4), int32 kv head h, then the K record
//          (9216 / 8704 bytes), then the packed query of one token (the stride
//          of 32 query heads: 4864 bytes)
//     out: float32 [128][8]
// Prints "ok" and exits 0 when the kernel ran and its wait completed.
#include <cstdio>
#include <cstdint>
#include <vector>

#include "bd_device.cuh"

using namespace bd;

namespace {

constexpr int kHq = 32;

// One page through lane quarter w = h % 4 of a 128-column score buffer: the
// query operand is the decode's zero image (28 groups of 512 B, group 12 =
// term 1 rows of heads 0..3, group 13 = term 2) offset by 4 w groups, the K
// record is the B operand (N = 128 tokens), the query's scale factors go to
// TMEM column 128 (+16), the record's to 160 (+16); warp w reads the quarter
// with the 16x256b load the decode uses.
__global__ void __launch_bounds__(128, 1) qk_page(const uint8_t* rec, const uint8_t* qp, int fmt, int h, float* out,
                                                 int* status) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ uint32_t tbase;
    __shared__ __align__(8) unsigned long long done;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = fmt == 0 ? 9216 : 8704;
    const int wq = h & 3;
    uint8_t* Ks = sm;               // the record, as the decode's K ring slot holds it
    uint8_t* Qi = sm + 9216;        // query image, 28 x 512 B
    uint8_t* Sf = Qi + 28 * 512;    // the query's scale-factor groups, 2 x 512 B
    if (warp == 0) tmem_alloc(smem_u32(&tbase), 256);
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&done), 1);
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < rb / 16; i += 128)
        reinterpret_cast<uint4*>(Ks)[i] = reinterpret_cast<const uint4*>(rec)[i];
    for (int i = threadIdx.x; i < (28 * 512 + 1024) / 16; i += 128)
        reinterpret_cast<uint4*>(Qi)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    if (threadIdx.x < 32) {
        const int row = lane >> 2, ch = lane & 3;
        const int term = row >> 2, hh = row & 3, jq = 4 * h + hh;
        *reinterpret_cast<uint4*>(Qi + (12 + term) * 512 + ch * 128 + hh * 16) =
            *reinterpret_cast<const uint4*>(qp + (term * kHq + jq) * 64 + 16 * ch);
        if (lane < 8) {
            // lane = (term st, head sh): A row line = sh (term 1) or 8 + sh (term 2)
            const int st = lane >> 2, sh = lane & 3, jr = 4 * h + sh;
            const int line = (st == 0 ? 0 : 8) + sh;
            if (fmt == 0) {
                const uint2 s = *reinterpret_cast<const uint2*>(qp + 2 * kHq * 64 + (st * kHq + jr) * 8);
                *reinterpret_cast<uint4*>(Sf + 16 * line) = make_uint4(s.x, s.x, s.x, s.x);
                *reinterpret_cast<uint4*>(Sf + 512 + 16 * line) = make_uint4(s.y, s.y, s.y, s.y);
            } else {
                const uint32_t s = *reinterpret_cast<const uint32_t*>(qp + 2 * kHq * 64 + (st * kHq + jr) * 4);
                *reinterpret_cast<uint4*>(Sf + 16 * line) = make_uint4(s, s, s, s);
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tbase;
    if (threadIdx.x == 0) {
        const int groups = fmt == 0 ? 2 : 1;
        for (int j = 0; j < groups; ++j) {
            tmem_cp_sf(tm + 128 + 16 * j, smem_u32(Sf + 512 * j));
            tmem_cp_sf(tm + 160 + 16 * j, smem_u32(Ks + kCodeBytes + 512 * j));
        }
        const uint32_t qimg = smem_u32(Qi + 12 * 512) - 4 * wq * 512;
        for (int j = 0; j < 2; ++j) {
            const uint64_t ad = smem_desc(qimg + 256 * j, 128, 512);
            const uint64_t bd = smem_desc(smem_u32(Ks) + 256 * j, 128, 512);
            if (fmt == 0)
                mma_nvf4(tm, ad, bd, mma_idesc_e2m1(128, false, 0), tm + 128 + 16 * j, tm + 160 + 16 * j, j);
            else
                mma_mxf4(tm, ad, bd, mma_idesc_e2m1(128, true, 2 * j), tm + 128, tm + 160, j);
        }
        tc_commit(smem_u32(&done));
    }
    const bool ok = mbar_wait_bounded(smem_u32(&done), 0, 1000000000ull, nullptr);
    tc_fence_after();
    if (!ok) {
        if (threadIdx.x == 0) *status = 1;
    } else if (warp == wq) {
        uint32_t r[64];
        tmem_ld_16x256b_x16(tm + ((uint32_t)(32 * warp) << 16), r);
        const int g = lane >> 2, t = lane & 3;
        if (g < 4) {
            for (int j = 0; j < 16; ++j)
                for (int e = 0; e < 2; ++e) {
                    const int tok = 8 * j + 2 * t + e;
                    out[tok * 8 + 2 * g] = __uint_as_float(r[4 * j + e]);          // term 1
                    out[tok * 8 + 2 * g + 1] = __uint_as_float(r[4 * j + 2 + e]);  // term 2
                }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, 256);
    }
}

}  // namespace

int main(int argc, char** argv) {
    if (argc != 3) return 2;
    FILE* f = std::fopen(argv[1], "rb");
    if (!f) return 2;
    int32_t hdr[2];
    if (std::fread(hdr, 4, 2, f) != 2) return 2;
    const int fmt = hdr[0], h = hdr[1];
    const int rb = fmt == 0 ? 9216 : 8704;
    const int qstride = 4864;
    if ((fmt != 0 && fmt != 1) || h < 0 || h >= kHq / 4) return 2;
    std::vector<uint8_t> rec(rb), qp(qstride);
    if (std::fread(rec.data(), 1, rb, f) != (size_t)rb || std::fread(qp.data(), 1, qstride, f) != (size_t)qstride)
        return 2;
    std::fclose(f);
    uint8_t *d_rec = nullptr, *d_qp = nullptr;
    float* d_out = nullptr;
    int* d_status = nullptr;
    if (cudaMalloc(&d_rec, 9216) != cudaSuccess || cudaMalloc(&d_qp, qstride) != cudaSuccess ||
        cudaMalloc(&d_out, 128 * 8 * 4) != cudaSuccess || cudaMalloc(&d_status, 4) != cudaSuccess)
        return 2;
    cudaMemset(d_rec, 0, 9216);
    cudaMemcpy(d_rec, rec.data(), rb, cudaMemcpyHostToDevice);
    cudaMemcpy(d_qp, qp.data(), qstride, cudaMemcpyHostToDevice);
    cudaMemset(d_status, 0, 4);
    const int smem = 9216 + 28 * 512 + 1024;
    cudaFuncSetAttribute(qk_page, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    qk_page<<<1, 128, smem>>>(d_rec, d_qp, fmt, h, d_out, d_status);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        std::printf("cuda error %s\n", cudaGetErrorString(e));
        return 2;
    }
    int status = 0;
    std::vector<float> out(128 * 8);
    cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(out.data(), d_out, out.size() * 4, cudaMemcpyDeviceToHost);
    if (status) {
        std::printf("wait timed out\n");
        return 2;
    }
    f = std::fopen(argv[2], "wb");
    if (!f || std::fwrite(out.data(), 4, out.size(), f) != out.size()) return 2;
    std::fclose(f);
    std::printf("ok\n");
    return 0;
}
