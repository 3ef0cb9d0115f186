// Two-term FP4 quantization of one token's query, shared by the standalone
// query kernel (bd_query.cu) and the decode kernel's fused path.
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
// Work item it = (query head it / 8, 16-dim chunk it % 8); the eight items of
// a head sit in eight consecutive lanes, where the Hadamard transform and the
// block quantization match the key writer lane for lane.  The two amax
// reductions span all participating threads.
#pragma once

#include "bd_device.cuh"
#include "bd_internal.h"

namespace bd {
namespace qquant {

constexpr unsigned kQFull = 0xFFFFFFFFu;

// Maximum of non-negative values over nthr threads tid = 0..nthr-1 (nthr a
// multiple of 32): their IEEE bit patterns order like the values, so one
// integer warp reduction replaces a shuffle chain; sync() is the group's
// barrier (red is reused from one call to the next).
template <class Sync>
__device__ __forceinline__ float group_max(float v, float* red, int tid, int nthr, Sync sync) {
    v = __uint_as_float(__reduce_max_sync(kQFull, __float_as_uint(v)));
    const int warp = tid >> 5, nw = nthr >> 5;
    sync();
    if ((tid & 31) == 0) red[warp] = v;
    sync();
    float r = 0.0f;
    for (int w = 0; w < nw; ++w) r = fmaxf(r, red[w]);
    return r;
}

// One term: quantize this lane's 16 values, held as pairs xp[i] = (x[2i],
// x[2i+1]) (NVFP4: a whole block; MXFP4: half of a 32-block shared with lane
// c^1), store codes and scale bytes (when `store`) and return the
// reconstruction in xh.  z: the run-time -0.0f of mulz2 in both lanes.
__device__ __forceinline__ void quant_term(const QueryArgs& a, const float2* xp, float g, float2 z, uint8_t* qp,
                                           int term, int j, int c, float2* xh, bool store) {
    const int hq = a.hq;
    uint32_t w0 = 0, w1 = 0, sb;
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(xp[i].x), fabsf(xp[i].y)));
    float2 S2;
    if (a.format == BD_FORMAT_NVFP4) {
        const float t = __fmul_rn(6.0f, g);
        const float s = __fdiv_rn(amax, t);
        sb = e4m3(s);
        const float S = __fmul_rn(e4m3_value(sb), g);
        const float inv = __frcp_rn(S);
        const bool zero = (S == 0.0f) || isinf(inv);
        const float2 inv2 = splat2(inv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 q = mul2(xp[i], inv2);
            const uint32_t byte = e2m1x2(q.x, q.y);
            if (i < 4) w0 |= byte << (8 * i);
            else w1 |= byte << (8 * (i - 4));
        }
        if (zero) {   // codes 0, so x_hat = +0 * S = +0
            w0 = 0;
            w1 = 0;
        }
        S2 = splat2(S);
        if (store) qp[2 * hq * 64 + (term * hq + j) * 8 + c] = (uint8_t)sb;
    } else {
        const float amax32 = fmaxf(amax, __shfl_xor_sync(kQFull, amax, 1));
        const int E = ilog2f(amax32 == 0.0f ? 1.0f : amax32);
        const int ea = min(127, max(-127, E - 2)), eb = min(127, max(-127, E - 1));
        float sse[2];
        uint32_t ca0, ca1, cb0, cb1;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            float2 wp[8];
            if (k == 0) mx_enc_err16x2(xp, ea, z, ca0, ca1, wp);
            else mx_enc_err16x2(xp, eb, z, cb0, cb1, wp);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                wp[i] = add2(wp[i], make_float2(__shfl_xor_sync(kQFull, wp[i].x, 1), __shfl_xor_sync(kQFull, wp[i].y, 1)));
            sse[k] = tree16x2(wp);
        }
        const bool zero = amax32 == 0.0f;   // codes 0 and x_hat = +0
        const bool pickb = sse[1] < sse[0];
        const int e = pickb ? eb : ea;
        w0 = zero ? 0u : (pickb ? cb0 : ca0);
        w1 = zero ? 0u : (pickb ? cb1 : ca1);
        S2 = splat2(pow2i(e));
        sb = zero ? 0u : (uint32_t)(e + 127);
        if (store && !(c & 1)) qp[2 * hq * 64 + (term * hq + j) * 4 + (c >> 1)] = (uint8_t)sb;
    }
    // x_hat = value(code) * S, rounded once per element
    uint32_t hv[8];
    e2m1x8_to_f16x2x4(w0, hv);
    e2m1x8_to_f16x2x4(w1, hv + 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) xh[i] = mulz2(f16x2_to_float2(hv[i]), S2, z);
    if (store) *reinterpret_cast<uint2*>(qp + (term * hq + j) * 64 + 8 * c) = make_uint2(w0, w1);
}

// Quantize the token whose raw query is qt (bf16 [hq][128]) into the packed
// record qp (a.stride bytes, global or shared memory), by nthr threads
// tid = 0..nthr-1, each taking the NI items it = tid + nthr i; items past
// hq * 8 compute on zeros (they take part in the shuffles) and store
// nothing.  mu: the layer's key mean [Hkv][128] (read only with centering).
// The second term's codes and scale bytes, and q.mu, are produced only for
// query heads j in [j2_lo, j2_hi) (both per-tensor scales still cover every
// head); a caller that restricts them keeps each warp's heads all in or all
// out.  mu_pre.ok: mu_pre.v holds this thread's 16 key-mean values
// (mu[j / 4][16 c .. 16 c + 15] of its single item, NI = 1), loaded by the
// caller ahead of time; otherwise they are read from mu here.
struct MuPre {
    float4 v[4];
    bool ok;
};

template <int NI, class Sync>
__device__ void quantize_token(const QueryArgs& a, const uint16_t* qt, const float* mu, uint8_t* qp, int tid, int nthr,
                               float* red, Sync sync, int j2_lo = 0, int j2_hi = 1 << 30,
                               MuPre mu_pre = MuPre{}) {
    const int hq = a.hq;
    const int c = tid & 7;
    const float2 z = splat2(a.zero_addend);
    float2 x[NI][8];   // the item's 16 values as pairs (2i, 2i+1)
    float qmu[NI];
    bool act[NI];
    int jh[NI];
#pragma unroll
    for (int n = 0; n < NI; ++n) {
        const int it = tid + nthr * n;
        act[n] = it < hq * 8;
        jh[n] = it >> 3;
        if (act[n]) {
            const uint16_t* src = qt + (size_t)jh[n] * kD + 16 * c;
            uint4 u0 = *reinterpret_cast<const uint4*>(src);
            uint4 u1 = *reinterpret_cast<const uint4*>(src + 8);
            const uint32_t wd[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) x[n][i] = make_float2(bf16_lo(wd[i]), bf16_hi(wd[i]));
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[n][i] = make_float2(0.0f, 0.0f);
        }
        // q.mu on the unrotated query (fp32, lane-partial then a 3-step butterfly)
        qmu[n] = 0.0f;
        if (a.centering && mu && act[n] && jh[n] >= j2_lo && jh[n] < j2_hi) {
            const float4* m4 = reinterpret_cast<const float4*>(mu + (jh[n] / kGroup) * kD + 16 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v = (NI == 1 && mu_pre.ok) ? mu_pre.v[i] : m4[i];
                qmu[n] = fmaf(x[n][2 * i].x, v.x, qmu[n]);
                qmu[n] = fmaf(x[n][2 * i].y, v.y, qmu[n]);
                qmu[n] = fmaf(x[n][2 * i + 1].x, v.z, qmu[n]);
                qmu[n] = fmaf(x[n][2 * i + 1].y, v.w, qmu[n]);
            }
        }
        qmu[n] += __shfl_xor_sync(kQFull, qmu[n], 1);
        qmu[n] += __shfl_xor_sync(kQFull, qmu[n], 2);
        qmu[n] += __shfl_xor_sync(kQFull, qmu[n], 4);

        if (a.rotation) {
            // stride 1 inside each pair
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float u = x[n][i].x, v = x[n][i].y;
                x[n][i] = make_float2(__fadd_rn(u, v), __fsub_rn(u, v));
            }
            // strides 2, 4, 8 between pairs
#pragma unroll
            for (int hs = 1; hs < 8; hs <<= 1)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (!(i & hs)) {
                        const float2 u = x[n][i], v = x[n][i + hs];
                        x[n][i] = add2(u, v);
                        x[n][i + hs] = sub2(u, v);
                    }
#pragma unroll
            for (int m = 1; m <= 4; m <<= 1) {
                // p - x in the upper lane, x + p in the lower one: fma(x, +-1, p)
                // rounds the exact p +- x once, like the add or subtract
                const float2 sgn = splat2((c & m) ? -1.0f : 1.0f);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 p = make_float2(__shfl_xor_sync(kQFull, x[n][i].x, m),
                                                 __shfl_xor_sync(kQFull, x[n][i].y, m));
                    x[n][i] = fma2(x[n][i], sgn, p);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) x[n][i] = mulz2(x[n][i], splat2(kRot), z);
        }
    }

    float amax = 0.0f;
#pragma unroll
    for (int n = 0; n < NI; ++n)
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(x[n][i].x), fabsf(x[n][i].y)));
    amax = group_max(amax, red, tid, nthr, sync);
    float g1 = 1.0f;
    if (a.format == BD_FORMAT_NVFP4 && amax != 0.0f) g1 = __fdiv_rn(amax, 2688.0f);
    float2 xh[NI][8];
#pragma unroll
    for (int n = 0; n < NI; ++n) quant_term(a, x[n], g1, z, qp, 0, jh[n], c, xh[n], act[n]);

    float g2 = 0.0f;
    if (a.terms == 2) {
        float amax_r = 0.0f;
#pragma unroll
        for (int n = 0; n < NI; ++n)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                x[n][i] = sub2(x[n][i], xh[n][i]);
                amax_r = fmaxf(amax_r, fmaxf(fabsf(x[n][i].x), fabsf(x[n][i].y)));
            }
        amax_r = group_max(amax_r, red, tid, nthr, sync);
        g2 = 1.0f;
        if (a.format == BD_FORMAT_NVFP4 && amax_r != 0.0f) g2 = __fdiv_rn(amax_r, 2688.0f);
#pragma unroll
        for (int n = 0; n < NI; ++n)
            if (jh[n] >= j2_lo && jh[n] < j2_hi) quant_term(a, x[n], g2, z, qp, 1, jh[n], c, xh[n], act[n]);
    } else {
#pragma unroll
        for (int n = 0; n < NI; ++n) {
            if (!act[n]) continue;
            const int j = jh[n];
            *reinterpret_cast<uint2*>(qp + (hq + j) * 64 + 8 * c) = make_uint2(0u, 0u);
            if (a.format == BD_FORMAT_NVFP4) qp[2 * hq * 64 + (hq + j) * 8 + c] = 0;
            else if (!(c & 1)) qp[2 * hq * 64 + (hq + j) * 4 + (c >> 1)] = 0;
        }
    }

    const int goff = 2 * hq * 64 + 2 * hq * 8;
    if (tid == 0) {
        reinterpret_cast<float*>(qp + goff)[0] = g1;
        reinterpret_cast<float*>(qp + goff)[1] = g2;
        reinterpret_cast<float*>(qp + goff)[2] = 0.0f;
        reinterpret_cast<float*>(qp + goff)[3] = 0.0f;
    }
#pragma unroll
    for (int n = 0; n < NI; ++n)
        if (act[n] && c == 0 && jh[n] >= j2_lo && jh[n] < j2_hi) reinterpret_cast<float*>(qp + goff + 16)[jh[n]] = qmu[n];
    // zero the bytes no field covers: the unused half of the scale area in
    // MXFP4 and the tail after q.mu
    if (a.format == BD_FORMAT_MXFP4)
        for (int i = tid; i < 2 * hq * 4; i += nthr) qp[2 * hq * 64 + 2 * hq * 4 + i] = 0;
    for (size_t i = goff + 16 + 4 * hq + tid; i < a.stride; i += nthr) qp[i] = 0;
}

}  // namespace qquant
}  // namespace bd
