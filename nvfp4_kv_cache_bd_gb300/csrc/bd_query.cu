// Two-term FP4 query quantization.
//
// Method: BitDecoding-FP4 evaluation config (config.py) RECIPE
// dual_residual_query_quantization with nvfp4_query_terms = 2, query scale
// mode "amax6", Hadamard rotation (nvfp4_rotation); MXFP4 queries use the
// "mxfp4_search" rule.  Per token: q -> rotate -> Q1 (per-tensor scale
// g1 = amax/2688 over the token's Hq*128 values) -> R = q_rot - Q1hat -> Q2
// (g2 = amax(R)/2688); a zero amax gives g = 1.  Also stores q.mu (unrotated
// bf16 q times the layer's key mean, fp32) so the decode can restore the key
// mean's contribution to the FP4 logits.
//
// One CTA per token, one thread per (query head j, 16-dim chunk c): the
// Hadamard transform and block quantization match the key writer lane for
// lane; the two amax reductions span the CTA.
#include "bd_device.cuh"

namespace bd {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

// CTA-wide maximum of non-negative values: their IEEE bit patterns order
// like the values, so one integer warp reduction replaces a shuffle chain.
__device__ __forceinline__ float block_max(float v, float* red) {
    v = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(v)));
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[warp] = v;
    __syncthreads();
    float r = 0.0f;
    for (int w = 0; w < nw; ++w) r = fmaxf(r, red[w]);
    return r;
}

// One term: quantize this lane's 16 values x (NVFP4: a whole block; MXFP4:
// half of a 32-block shared with lane c^1), store codes and scale bytes and
// return the reconstruction in xh.
__device__ __forceinline__ void quant_term(const QueryArgs& a, const float* x, float g, uint8_t* qp, int term,
                                           int j, int c, float* xh) {
    const int hq = a.hq;
    uint32_t w0 = 0, w1 = 0, sb;
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    if (a.format == BD_FORMAT_NVFP4) {
        const float t = __fmul_rn(6.0f, g);
        const float s = __fdiv_rn(amax, t);
        sb = e4m3(s);
        const float S = __fmul_rn(e4m3_value(sb), g);
        const float inv = __frcp_rn(S);
        const bool zero = (S == 0.0f) || isinf(inv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t byte = zero ? 0u : e2m1x2(__fmul_rn(x[2 * i], inv), __fmul_rn(x[2 * i + 1], inv));
            if (i < 4) w0 |= byte << (8 * i);
            else w1 |= byte << (8 * (i - 4));
            float2 val = f16x2_to_float2(e2m1x2_to_f16x2(byte));
            xh[2 * i] = zero ? 0.0f : __fmul_rn(val.x, S);
            xh[2 * i + 1] = zero ? 0.0f : __fmul_rn(val.y, S);
        }
        qp[2 * hq * 64 + (term * hq + j) * 8 + c] = (uint8_t)sb;
    } else {
        const float amax32 = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
        const int E = ilog2f(amax32 == 0.0f ? 1.0f : amax32);
        const int ea = min(127, max(-127, E - 2)), eb = min(127, max(-127, E - 1));
        float sse[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int e = k ? eb : ea;
            const float down = pow2i(-e), up = pow2i(e);
            float w[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t byte = e2m1x2(__fmul_rn(x[2 * i], down), __fmul_rn(x[2 * i + 1], down));
                float2 val = f16x2_to_float2(e2m1x2_to_f16x2(byte));
                float e0 = __fsub_rn(x[2 * i], __fmul_rn(val.x, up));
                float e1 = __fsub_rn(x[2 * i + 1], __fmul_rn(val.y, up));
                w[2 * i] = __fmul_rn(e0, e0);
                w[2 * i + 1] = __fmul_rn(e1, e1);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __fadd_rn(w[i], __shfl_xor_sync(kFull, w[i], 1));
#pragma unroll
            for (int hh = 8; hh >= 1; hh >>= 1)
#pragma unroll
                for (int i = 0; i < hh; ++i) w[i] = __fadd_rn(w[i], w[i + hh]);
            sse[k] = w[0];
        }
        const bool zero = amax32 == 0.0f;
        const int e = (sse[1] < sse[0]) ? eb : ea;
        const float down = pow2i(-e), up = pow2i(e);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t byte = zero ? 0u : e2m1x2(__fmul_rn(x[2 * i], down), __fmul_rn(x[2 * i + 1], down));
            if (i < 4) w0 |= byte << (8 * i);
            else w1 |= byte << (8 * (i - 4));
            float2 val = f16x2_to_float2(e2m1x2_to_f16x2(byte));
            xh[2 * i] = zero ? 0.0f : __fmul_rn(val.x, up);
            xh[2 * i + 1] = zero ? 0.0f : __fmul_rn(val.y, up);
        }
        sb = zero ? 0u : (uint32_t)(e + 127);
        if (!(c & 1)) qp[2 * hq * 64 + (term * hq + j) * 4 + (c >> 1)] = (uint8_t)sb;
    }
    *reinterpret_cast<uint2*>(qp + (term * hq + j) * 64 + 8 * c) = make_uint2(w0, w1);
}

__global__ void __launch_bounds__(512) query_kernel(const QueryArgs a) {
    __shared__ float red[16];
    const int b = blockIdx.x;
    const int j = threadIdx.x >> 3, c = threadIdx.x & 7;
    const int hq = a.hq;
    uint8_t* qp = a.qp + (size_t)b * a.stride;
    // The layer's key mean is context state written only by the synchronous
    // bd_set_key_shift, never by a kernel: it is read before the wait below.
    float4 mu4[4] = {};
    if (a.centering && a.mu) {
        const float4* mu = reinterpret_cast<const float4*>(a.mu + (j / kGroup) * kD + 16 * c);
#pragma unroll
        for (int i = 0; i < 4; ++i) mu4[i] = mu[i];
    }
    // Programmatic dependent launch: let the dependent decode launch at once
    // (it streams the layer's static FP4 pages and waits for this grid before
    // it reads the packed query), then wait for the grid that precedes us in
    // the stream, whose outputs may feed q.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");

    float x[16];
    {
        const uint16_t* src = a.q + ((size_t)b * hq + j) * kD + 16 * c;
        uint4 u0 = *reinterpret_cast<const uint4*>(src);
        uint4 u1 = *reinterpret_cast<const uint4*>(src + 8);
        const uint32_t wd[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x[2 * i] = bf16_lo(wd[i]);
            x[2 * i + 1] = bf16_hi(wd[i]);
        }
    }
    // q.mu on the unrotated query (fp32, lane-partial then a 3-step butterfly)
    float qmu = 0.0f;
    if (a.centering && a.mu) {
        const float mu[16] = {mu4[0].x, mu4[0].y, mu4[0].z, mu4[0].w, mu4[1].x, mu4[1].y, mu4[1].z, mu4[1].w,
                              mu4[2].x, mu4[2].y, mu4[2].z, mu4[2].w, mu4[3].x, mu4[3].y, mu4[3].z, mu4[3].w};
#pragma unroll
        for (int i = 0; i < 16; ++i) qmu = fmaf(x[i], mu[i], qmu);
    }
    qmu += __shfl_xor_sync(kFull, qmu, 1);
    qmu += __shfl_xor_sync(kFull, qmu, 2);
    qmu += __shfl_xor_sync(kFull, qmu, 4);

    if (a.rotation) {
#pragma unroll
        for (int hs = 1; hs < 16; hs <<= 1)
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (!(i & hs)) {
                    float u = x[i], v = x[i + hs];
                    x[i] = __fadd_rn(u, v);
                    x[i + hs] = __fsub_rn(u, v);
                }
#pragma unroll
        for (int m = 1; m <= 4; m <<= 1) {
            // p - x in the upper lane, x + p in the lower one: fma(x, +-1, p)
            // rounds the exact p +- x once, like the add or subtract
            const float sgn = (c & m) ? -1.0f : 1.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float p = __shfl_xor_sync(kFull, x[i], m);
                x[i] = __fmaf_rn(x[i], sgn, p);
            }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = __fmul_rn(x[i], kRot);
    }

    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = block_max(amax, red);
    float g1 = 1.0f;
    if (a.format == BD_FORMAT_NVFP4 && amax != 0.0f) g1 = __fdiv_rn(amax, 2688.0f);
    float xh[16];
    quant_term(a, x, g1, qp, 0, j, c, xh);

    float g2 = 0.0f;
    if (a.terms == 2) {
        float amax_r = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            x[i] = __fsub_rn(x[i], xh[i]);
            amax_r = fmaxf(amax_r, fabsf(x[i]));
        }
        amax_r = block_max(amax_r, red);
        g2 = 1.0f;
        if (a.format == BD_FORMAT_NVFP4 && amax_r != 0.0f) g2 = __fdiv_rn(amax_r, 2688.0f);
        quant_term(a, x, g2, qp, 1, j, c, xh);
    } else {
        *reinterpret_cast<uint2*>(qp + (hq + j) * 64 + 8 * c) = make_uint2(0u, 0u);
        if (a.format == BD_FORMAT_NVFP4) qp[2 * hq * 64 + (hq + j) * 8 + c] = 0;
        else if (!(c & 1)) qp[2 * hq * 64 + (hq + j) * 4 + (c >> 1)] = 0;
    }

    const int goff = 2 * hq * 64 + 2 * hq * 8;
    if (threadIdx.x == 0) {
        reinterpret_cast<float*>(qp + goff)[0] = g1;
        reinterpret_cast<float*>(qp + goff)[1] = g2;
        reinterpret_cast<float*>(qp + goff)[2] = 0.0f;
        reinterpret_cast<float*>(qp + goff)[3] = 0.0f;
    }
    if (c == 0) reinterpret_cast<float*>(qp + goff + 16)[j] = qmu;
    // zero the bytes no field covers: the unused half of the scale area in
    // MXFP4 and the tail after q.mu
    if (a.format == BD_FORMAT_MXFP4)
        for (int i = threadIdx.x; i < 2 * hq * 4; i += blockDim.x) qp[2 * hq * 64 + 2 * hq * 4 + i] = 0;
    for (size_t i = goff + 16 + 4 * hq + threadIdx.x; i < a.stride; i += blockDim.x) qp[i] = 0;
}

}  // namespace

cudaError_t launch_query(const QueryArgs& a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.B);
    cfg.blockDim = dim3((unsigned)(a.hq * 8));
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, query_kernel, a);
}

}  // namespace bd
