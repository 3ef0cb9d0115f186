// Paged single-token decode attention over the hybrid cache (BF16 sink +
// packed FP4 pages + BF16 tail), flash-decoding style split-K over pages,
// and the split combine.
//
// Method: "How openbitsys/bitdecoding-fp4 works" (decode interface -> paged
// attention kernel; hybrid cache); BitDecoding-FP4 evaluation config
// (config.py): KV_MODES sink_tokens 16, PARITY_ENGINE_KWARGS block_size 128,
// probability_environment ("amax6" / "amax2_or_amax6" with c in {1, 8} and
// tau in [0, 448]), RECIPE dual_residual_query_quantization (two query terms).
//
// Grid (nsplit + 1, kv heads, sequences).  Split 0 of a (sequence, kv head)
// handles the BF16 sink and tail tokens with exact probabilities; splits
// 1..nsplit each stream a contiguous range of that sequence's FP4 pages.
//
// FP4 split CTA: warp 4 is the producer; one elected lane streams each
// page's K and V records (9216 B each in NVFP4) into a 4-stage shared-memory
// ring with cp.async.bulk, completing on per-stage "full" mbarriers; warps
// 0..3 consume.  Consumer warp w owns tokens 32w..32w+31 of every page:
//  QK  : m16n8k16 f16 MMAs, M = 16 tokens, N = 8 = 4 query heads x 2 query
//        terms, K = 16 head dims.  FP4 codes are widened by cvt e2m1x2->f16x2
//        and multiplied by their E4M3 scale in f16, which is exact
//        (E2M1 x E4M3 has at most 6 significant bits and lies in
//        [2^-10, 2688]); the query terms are exact the same way.  Per-tensor
//        scales, the 1/sqrt(128) softmax scale and q.mu are applied to the
//        fp32 accumulators.
//  P   : per page, the page maximum m_p of every head (the four warps trade
//        their maxima through shared memory at one named barrier); P =
//        exp(s - m_p); each 16-token block is quantized to FP4 with the
//        amax2-or-amax6 rule; Phat = E2M1 x E4M3 / c is again exact in f16.
//  PV  : O^T[128 dims][8] += Vhat^T[dims][16 tokens] Phat^T, V codes widened
//        and scaled exactly as for K.  The V record stores tokens tau and
//        tau+8 in one byte, which is exactly an A-fragment register of this
//        MMA; Phat reaches the B-fragment layout with two warp shuffles.
//  The page partial (m_p, l_p, O_p) is merged into a running (M, L, O) per
//  warp; at the end the four warps' partials are summed through shared
//  memory and written to the workspace.
// The combine kernel merges all splits: O = sum e^(m-M) O / sum e^(m-M) l.
#include <math.h>

#include "bd_device.cuh"

namespace bd {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kStages = 4;
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kMaxRec = 9216;
constexpr int kStageBytes = 2 * kMaxRec;
constexpr int kRingBytes = kStages * kStageBytes;
constexpr float kSmLog2e = 0.08838834764831845f * 1.4426950408889634f;  // log2(e)/sqrt(128)

struct Ctl {
    unsigned long long full[kStages];
    unsigned long long empty[kStages];
    float red[2][kConsumers][4];
    int vote[2][kConsumers];   // per page: 1 if that warp's wait for the page gave up
    int abort_flag;            // hint that lets pending waits give up early
    int issued;
    int consumed[kConsumers];
};
constexpr int kSmemBytes = kRingBytes + (int)sizeof(Ctl);

__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint32_t lds16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }

// 16-bit pair of code bytes (bytes 2k, 2k+1) from a 16-byte chunk.
__device__ __forceinline__ uint32_t byte_pair(const uint4& c, int k) {
    const uint32_t wd = (k < 2) ? c.x : (k < 4) ? c.y : (k < 6) ? c.z : c.w;
    return (k & 1) ? (wd >> 16) : (wd & 0xFFFFu);
}

// f16 bits of 2^k for k <= 0 (subnormal below -14, zero below -24).
__device__ __forceinline__ uint32_t f16_pow2(int k) {
    if (k >= -14) return (uint32_t)(k + 15) << 10;
    if (k >= -24) return 1u << (k + 24);
    return 0u;
}

__device__ __forceinline__ void write_empty(float* part, int nsplit1) {
    for (int hh = 0; hh < 4; ++hh) {
        part[hh * nsplit1 * kPartStride + 0] = -INFINITY;
        part[hh * nsplit1 * kPartStride + 1] = 0.0f;
    }
}

// ------------------------------------------------------ BF16 sink + tail --

__device__ void bf16_segment(const DecodeArgs& a, int b, int h, int L, float* part, uint8_t* smem) {
    const int ns = min(L, kSink);
    const int rest = max(0, L - kSink);
    const int npages = rest / kPage;
    const int nt = rest - npages * kPage;
    const int T = ns + nt;
    const int nsplit1 = a.nsplit + 1;
    const int tid = threadIdx.x;
    if (T == 0) {
        if (tid == 0) write_empty(part, nsplit1);
        return;
    }
    float* qf = reinterpret_cast<float*>(smem);      // [4][128]
    float* sp = qf + 4 * kD;                          // [4][144]
    float* mh = sp + 4 * 144;                         // [4]
    float* lh = mh + 4;                               // [4]
    for (int i = tid; i < 4 * kD; i += blockDim.x) {
        const uint16_t bits = a.q[((size_t)b * a.hq + 4 * h + i / kD) * kD + (i % kD)];
        qf[i] = __uint_as_float((uint32_t)bits << 16);
    }
    __syncthreads();
    auto krow = [&](int tau) -> const uint16_t* {
        return tau < ns ? a.sink_k + (((size_t)b * kSink + tau) * a.hkv + h) * kD
                        : a.tail_k + (((size_t)b * kPage + (tau - ns)) * a.hkv + h) * kD;
    };
    auto vrow = [&](int tau) -> const uint16_t* {
        return tau < ns ? a.sink_v + (((size_t)b * kSink + tau) * a.hkv + h) * kD
                        : a.tail_v + (((size_t)b * kPage + (tau - ns)) * a.hkv + h) * kD;
    };
    for (int tau = tid; tau < T; tau += blockDim.x) {
        const uint4* kr = reinterpret_cast<const uint4*>(krow(tau));
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        for (int c = 0; c < 16; ++c) {
            const uint4 u = kr[c];
            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float k0 = bf16_lo(wd[e]), k1 = bf16_hi(wd[e]);
                const int d = 8 * c + 2 * e;
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) s[hh] = fmaf(qf[hh * kD + d + 1], k1, fmaf(qf[hh * kD + d], k0, s[hh]));
            }
        }
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) sp[hh * 144 + tau] = s[hh] * kSmLog2e;
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < 4) {
        float m = -INFINITY;
        for (int tau = lane; tau < T; tau += 32) m = fmaxf(m, sp[warp * 144 + tau]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        float l = 0.0f;
        for (int tau = lane; tau < T; tau += 32) {
            const float p = ex2(sp[warp * 144 + tau] - m);
            sp[warp * 144 + tau] = p;
            l += p;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
        if (lane == 0) {
            mh[warp] = m;
            lh[warp] = l;
        }
    }
    __syncthreads();
    if (tid < kD) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int tau = 0; tau < T; ++tau) {
            const float v = __uint_as_float((uint32_t)vrow(tau)[tid] << 16);
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) acc[hh] = fmaf(sp[hh * 144 + tau], v, acc[hh]);
        }
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
            float* ph = part + hh * nsplit1 * kPartStride;
            ph[4 + tid] = acc[hh];
            if (tid == 0) {
                ph[0] = mh[hh];
                ph[1] = lh[hh];
            }
        }
    }
}

// --------------------------------------------------------- FP4 page split --

template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int L = a.seq_lens[b];
    const int nsplit1 = a.nsplit + 1;
    float* part = a.ws + ((size_t)(b * a.hq + 4 * h) * nsplit1 + split) * kPartStride;

    if (split == 0) {
        bf16_segment(a, b, h, L, part, smem);
        return;
    }
    // pages past the block-table row are ignored (the header bounds L)
    const int npages = min(max(0, L - kSink) / kPage, a.max_blocks);
    const int p0 = (split - 1) * a.pages_per_split;
    const int p1 = min(p0 + a.pages_per_split, npages);
    if (p0 >= p1) {
        if (threadIdx.x == 0) write_empty(part, nsplit1);
        return;
    }
    const int n = p1 - p0;
    constexpr int RB = (FMT == BD_FORMAT_NVFP4) ? 9216 : 8704;
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + kRingBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), kConsumers);
        }
        ctl->abort_flag = 0;
        ctl->issued = 0;
        fence_mbar_init();
    }
    if (threadIdx.x < kConsumers) ctl->consumed[threadIdx.x] = 0;
    __syncthreads();

    if (warp == kConsumers) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            const int32_t* bt = a.block_table + (size_t)b * a.max_blocks + p0;
            const size_t rec_stride = (size_t)RB;
            int k = 0;
            for (; k < n; ++k) {
                const int s = k % kStages;
                if (k >= kStages) {
                    if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ((k / kStages) - 1) & 1, kWaitLimitNs,
                                           &ctl->abort_flag)) {
                        if (!ctl->abort_flag) record_error(a.err, BD_ERR_TIMEOUT);
                        ctl->abort_flag = 1;
                        break;
                    }
                }
                const int64_t phys = bt[k];
                const uint8_t* krec = a.pool + ((phys * a.hkv + h) * 2) * rec_stride;
                const uint32_t full = smem_u32(&ctl->full[s]);
                const uint32_t dst = smem_u32(smem + s * kStageBytes);
                mbar_arrive_expect_tx(full, 2 * RB);
                bulk_g2s(dst, krec, RB, full);
                bulk_g2s(dst + kMaxRec, krec + RB, RB, full);
            }
            ctl->issued = k;
        }
    } else {
        // ------------------------------------------------------ consumers --
        const int g = lane >> 2, t = lane & 3;
        const uint8_t* qrec = a.qp + (size_t)b * a.qstride;
        const int hq = a.hq;
        // B fragments of the query: row n = g -> head 4h + g/2, term g%2;
        // this lane's k-slots are head dims 32t .. 32t+31.
        uint32_t qB[16];
        float qx[2];   // MXFP4: 2^(row reference exponent) of this lane's C columns
        {
            const int jq = 4 * h + (g >> 1), term = g & 1;
            const uint4 qc = *reinterpret_cast<const uint4*>(qrec + (term * hq + jq) * 64 + 16 * t);
            uint32_t slo, shi;
            if (FMT == BD_FORMAT_NVFP4) {
                const uint32_t qsd = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(
                    qrec + 2 * hq * 64 + (term * hq + jq) * 8 + 2 * t));
                slo = bcast_lo(qsd);
                shi = bcast_hi(qsd);
            } else {
                const uint32_t e4 = *reinterpret_cast<const uint32_t*>(qrec + 2 * hq * 64 + (term * hq + jq) * 4);
                int emax = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) emax = max(emax, (int)((e4 >> (8 * q)) & 0xFF));
                const int et = (int)((e4 >> (8 * t)) & 0xFF);
                slo = shi = bcast_lo(f16_pow2(et - emax));
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t pr = byte_pair(qc, kk);
                const uint32_t sc = kk < 4 ? slo : shi;
                qB[2 * kk] = hmul2(e2m1x2_to_f16x2(pr & 0xFF), sc);
                qB[2 * kk + 1] = hmul2(e2m1x2_to_f16x2(pr >> 8), sc);
            }
            if (FMT == BD_FORMAT_MXFP4) {
#pragma unroll
                for (int term2 = 0; term2 < 2; ++term2) {
                    const uint32_t e4 =
                        *reinterpret_cast<const uint32_t*>(qrec + 2 * hq * 64 + (term2 * hq + 4 * h + t) * 4);
                    int emax = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) emax = max(emax, (int)((e4 >> (8 * q)) & 0xFF));
                    qx[term2] = pow2i(emax - 127);
                }
            } else {
                qx[0] = qx[1] = 1.0f;
            }
        }
        const float* gq = reinterpret_cast<const float*>(qrec + 2 * hq * 64 + 2 * hq * 8);
        const float gK = (FMT == BD_FORMAT_NVFP4) ? a.gk : 1.0f;
        const float gV = (FMT == BD_FORMAT_NVFP4) ? a.gv : 1.0f;
        const float a1 = kSmLog2e * gK * ((FMT == BD_FORMAT_NVFP4) ? gq[0] : qx[0]);
        const float a2 = kSmLog2e * gK * ((FMT == BD_FORMAT_NVFP4) ? gq[1] : qx[1]);
        const float bq = a.centering ? kSmLog2e * gq[4 + 4 * h + t] : 0.0f;
        const int cc = (a.p_mode == BD_P_AMAX2_OR_AMAX6) ? a.p_c : 1;
        const float ccf = (float)cc;
        const uint32_t inv_cc = bcast_lo((uint32_t)__half_as_ushort(__float2half_rn(1.0f / ccf)));

        float M[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float o[8][4];
#pragma unroll
        for (int bm = 0; bm < 8; ++bm) o[bm][0] = o[bm][1] = o[bm][2] = o[bm][3] = 0.0f;
        float lacc = 0.0f;

        int k = 0;
        for (; k < n; ++k) {
            const int s = k % kStages;
            const bool ok =
                mbar_wait_bounded(smem_u32(&ctl->full[s]), (k / kStages) & 1, kWaitLimitNs, &ctl->abort_flag);
            if (!ok) {
                if (!ctl->abort_flag) record_error(a.err, BD_ERR_TIMEOUT);
                ctl->abort_flag = 1;
            }
            const uint8_t* Ks = smem + s * kStageBytes;
            const uint8_t* Vs = Ks + kMaxRec;

            // ---------------- QK: scores (log2 units) for head t, tokens
            // 32w + 16 mi + g (+8)
            float sc[2][2];
#pragma unroll
            for (int mi = 0; mi < 2; ++mi) {
                const int tok0 = 16 * (2 * warp + mi) + g, tok1 = tok0 + 8;
                const uint4 c0 = lds128(Ks + tok0 * 64 + 16 * t);
                const uint4 c1 = lds128(Ks + tok1 * 64 + 16 * t);
                uint32_t s0lo, s0hi, s1lo, s1hi;
                float fk0 = 1.0f, fk1 = 1.0f;
                if (FMT == BD_FORMAT_NVFP4) {
                    const uint32_t sd0 = e4m3x2_to_f16x2(lds16(Ks + kCodeBytes + tok0 * 8 + 2 * t));
                    const uint32_t sd1 = e4m3x2_to_f16x2(lds16(Ks + kCodeBytes + tok1 * 8 + 2 * t));
                    s0lo = bcast_lo(sd0);
                    s0hi = bcast_hi(sd0);
                    s1lo = bcast_lo(sd1);
                    s1hi = bcast_hi(sd1);
                } else {
                    const int e0 = Ks[kCodeBytes + tok0 * 4 + t], e1 = Ks[kCodeBytes + tok1 * 4 + t];
                    int m0 = max(e0, __shfl_xor_sync(kFull, e0, 1));
                    m0 = max(m0, __shfl_xor_sync(kFull, m0, 2));
                    int m1 = max(e1, __shfl_xor_sync(kFull, e1, 1));
                    m1 = max(m1, __shfl_xor_sync(kFull, m1, 2));
                    s0lo = s0hi = bcast_lo(f16_pow2(e0 - m0));
                    s1lo = s1hi = bcast_lo(f16_pow2(e1 - m1));
                    fk0 = pow2i(m0 - 127);
                    fk1 = pow2i(m1 - 127);
                }
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t p0w = byte_pair(c0, kk), p1w = byte_pair(c1, kk);
                    const uint32_t sa = kk < 4 ? s0lo : s0hi, sb2 = kk < 4 ? s1lo : s1hi;
                    uint32_t A[4];
                    A[0] = hmul2(e2m1x2_to_f16x2(p0w & 0xFF), sa);
                    A[1] = hmul2(e2m1x2_to_f16x2(p1w & 0xFF), sb2);
                    A[2] = hmul2(e2m1x2_to_f16x2(p0w >> 8), sa);
                    A[3] = hmul2(e2m1x2_to_f16x2(p1w >> 8), sb2);
                    mma16816(acc, A, qB[2 * kk], qB[2 * kk + 1]);
                }
                sc[mi][0] = fmaf(fk0, fmaf(acc[1], a2, acc[0] * a1), bq);
                sc[mi][1] = fmaf(fk1, fmaf(acc[3], a2, acc[2] * a1), bq);
            }

            // ---------------- page maximum per head (all four warps)
            float mloc = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
            mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 4));
            mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 8));
            mloc = fmaxf(mloc, __shfl_xor_sync(kFull, mloc, 16));
            if (g == 0) ctl->red[k & 1][warp][t] = mloc;
            if (lane == 0) ctl->vote[k & 1][warp] = ok ? 0 : 1;
            named_bar_sync(1, kConsumers * 32);
            // every consumer warp reads the same four votes: the break is uniform
            if (ctl->vote[k & 1][0] | ctl->vote[k & 1][1] | ctl->vote[k & 1][2] | ctl->vote[k & 1][3]) break;
            float mp[4];
            {
                const float4 r0 = *reinterpret_cast<const float4*>(ctl->red[k & 1][0]);
                const float4 r1 = *reinterpret_cast<const float4*>(ctl->red[k & 1][1]);
                const float4 r2 = *reinterpret_cast<const float4*>(ctl->red[k & 1][2]);
                const float4 r3 = *reinterpret_cast<const float4*>(ctl->red[k & 1][3]);
                mp[0] = fmaxf(fmaxf(r0.x, r1.x), fmaxf(r2.x, r3.x));
                mp[1] = fmaxf(fmaxf(r0.y, r1.y), fmaxf(r2.y, r3.y));
                mp[2] = fmaxf(fmaxf(r0.z, r1.z), fmaxf(r2.z, r3.z));
                mp[3] = fmaxf(fmaxf(r0.w, r1.w), fmaxf(r2.w, r3.w));
            }
            const float mpt = (t == 0) ? mp[0] : (t == 1) ? mp[1] : (t == 2) ? mp[2] : mp[3];

            // ---------------- probabilities and their FP4 quantization
            uint32_t pv[2];
            float lpage = 0.0f;
#pragma unroll
            for (int mi = 0; mi < 2; ++mi) {
                const float p0 = ex2(sc[mi][0] - mpt), p1 = ex2(sc[mi][1] - mpt);
                lpage += p0 + p1;
                if (a.p_mode == BD_P_NONE) {
                    const __half2 hh = __floats2half2_rn(p0, p1);
                    pv[mi] = *reinterpret_cast<const uint32_t*>(&hh);
                } else {
                    const float u0 = p0 * ccf, u1 = p1 * ccf;
                    float am = fmaxf(u0, u1);
                    am = fmaxf(am, __shfl_xor_sync(kFull, am, 4));
                    am = fmaxf(am, __shfl_xor_sync(kFull, am, 8));
                    am = fmaxf(am, __shfl_xor_sync(kFull, am, 16));
                    const float mode = (a.p_mode == BD_P_AMAX2_OR_AMAX6 && am < a.tau) ? 2.0f : 6.0f;
                    const uint32_t sbyte = e4m3(__fdiv_rn(am, mode));
                    const uint32_t sdh = e4m3x2_to_f16x2(sbyte);
                    const float sd = __half2float(__ushort_as_half((unsigned short)(sdh & 0xFFFF)));
                    const float inv = __frcp_rn(sd);
                    const bool zero = (sd == 0.0f) || isinf(inv);
                    const uint32_t byte = zero ? 0u : e2m1x2(__fmul_rn(u0, inv), __fmul_rn(u1, inv));
                    pv[mi] = hmul2(e2m1x2_to_f16x2(byte), hmul2(bcast_lo(sdh), inv_cc));
                }
            }

            // ---------------- PV: O_p^T[dims][heads] for this warp's 32 tokens
            float op[8][4];
#pragma unroll
            for (int bm = 0; bm < 8; ++bm) op[bm][0] = op[bm][1] = op[bm][2] = op[bm][3] = 0.0f;
            float fv = 1.0f;    // MXFP4: 2^(reference exponent of this lane's V block)
            int ev_ref = 0;
            if (FMT == BD_FORMAT_MXFP4) {
                int em = 0;
#pragma unroll
                for (int mi = 0; mi < 2; ++mi) {
                    const int i = 2 * warp + mi;
                    const uint32_t e0 = lds16(Vs + kCodeBytes + ((i * 8 + t) * 4 + (g >> 1)) * 2);
                    const uint32_t e1 = lds16(Vs + kCodeBytes + ((i * 8 + t + 4) * 4 + (g >> 1)) * 2);
                    em = max(em, (int)max(max(e0 & 0xFF, e0 >> 8), max(e1 & 0xFF, e1 >> 8)));
                }
                em = max(em, __shfl_xor_sync(kFull, em, 1));
                em = max(em, __shfl_xor_sync(kFull, em, 2));
                em = max(em, __shfl_xor_sync(kFull, em, 4));
                ev_ref = em;
                fv = pow2i(em - 127);
            }
#pragma unroll
            for (int mi = 0; mi < 2; ++mi) {
                const int i = 2 * warp + mi;
                const int gs = g & 3;
                uint32_t b01 = __shfl_sync(kFull, pv[mi], 4 * t + gs);
                uint32_t b23 = __shfl_sync(kFull, pv[mi], 16 + 4 * t + gs);
                if (g >= 4) b01 = b23 = 0u;
                const uint4 v0 = lds128(Vs + (i * 8 + t) * kD + 16 * g);
                const uint4 v1 = lds128(Vs + (i * 8 + t + 4) * kD + 16 * g);
                uint32_t vs0, vs1;
                if (FMT == BD_FORMAT_NVFP4) {
                    vs0 = e4m3x2_to_f16x2(lds16(Vs + kCodeBytes + ((i * 8 + t) * 8 + g) * 2));
                    vs1 = e4m3x2_to_f16x2(lds16(Vs + kCodeBytes + ((i * 8 + t + 4) * 8 + g) * 2));
                } else {
                    const uint32_t e0 = lds16(Vs + kCodeBytes + ((i * 8 + t) * 4 + (g >> 1)) * 2);
                    const uint32_t e1 = lds16(Vs + kCodeBytes + ((i * 8 + t + 4) * 4 + (g >> 1)) * 2);
                    vs0 = f16_pow2((int)(e0 & 0xFF) - ev_ref) | (f16_pow2((int)(e0 >> 8) - ev_ref) << 16);
                    vs1 = f16_pow2((int)(e1 & 0xFF) - ev_ref) | (f16_pow2((int)(e1 >> 8) - ev_ref) << 16);
                }
#pragma unroll
                for (int bm = 0; bm < 8; ++bm) {
                    const uint32_t w0 = byte_pair(v0, bm), w1 = byte_pair(v1, bm);
                    uint32_t A[4];
                    A[0] = hmul2(e2m1x2_to_f16x2(w0 & 0xFF), vs0);
                    A[1] = hmul2(e2m1x2_to_f16x2(w0 >> 8), vs0);
                    A[2] = hmul2(e2m1x2_to_f16x2(w1 & 0xFF), vs1);
                    A[3] = hmul2(e2m1x2_to_f16x2(w1 >> 8), vs1);
                    mma16816(op[bm], A, b01, b23);
                }
            }
            // release the stage: every lane's shared-memory reads are done
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->empty[s]));

            // ---------------- merge the page into the running state
            float al[4], be[4];
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                const float mn = fmaxf(M[hh], mp[hh]);
                al[hh] = ex2(M[hh] - mn);
                be[hh] = ex2(mp[hh] - mn);
                M[hh] = mn;
            }
            // this lane's O columns are heads 2t, 2t+1 (t >= 2: padding columns)
            const bool odd = (t & 1) != 0;
            const float aA = odd ? al[2] : al[0], aB = odd ? al[3] : al[1];
            const float bA = (odd ? be[2] : be[0]) * gV * fv, bB = (odd ? be[3] : be[1]) * gV * fv;
#pragma unroll
            for (int bm = 0; bm < 8; ++bm) {
                o[bm][0] = fmaf(o[bm][0], aA, bA * op[bm][0]);
                o[bm][1] = fmaf(o[bm][1], aB, bB * op[bm][1]);
                o[bm][2] = fmaf(o[bm][2], aA, bA * op[bm][2]);
                o[bm][3] = fmaf(o[bm][3], aB, bB * op[bm][3]);
            }
            const float at = (t == 0) ? al[0] : (t == 1) ? al[1] : (t == 2) ? al[2] : al[3];
            const float bt2 = (t == 0) ? be[0] : (t == 1) ? be[1] : (t == 2) ? be[2] : be[3];
            lacc = fmaf(lacc, at, bt2 * lpage);
        }
        if (lane == 0) ctl->consumed[warp] = k;

        // ---------------- per-warp partials to shared memory
        __syncthreads();   // (A) every consumer is done with the ring
        float* sO = reinterpret_cast<float*>(smem);          // [4 warps][4 heads][128]
        float* sL = sO + kConsumers * 4 * kD;                // [4 warps][4 heads]
        if (t < 2) {
#pragma unroll
            for (int bm = 0; bm < 8; ++bm) {
                const int d = 16 * g + 2 * bm;
                sO[(warp * 4 + 2 * t) * kD + d] = o[bm][0];
                sO[(warp * 4 + 2 * t + 1) * kD + d] = o[bm][1];
                sO[(warp * 4 + 2 * t) * kD + d + 1] = o[bm][2];
                sO[(warp * 4 + 2 * t + 1) * kD + d + 1] = o[bm][3];
            }
        }
        lacc += __shfl_xor_sync(kFull, lacc, 4);
        lacc += __shfl_xor_sync(kFull, lacc, 8);
        lacc += __shfl_xor_sync(kFull, lacc, 16);
        if (g == 0) sL[warp * 4 + t] = lacc;
        named_bar_sync(1, kConsumers * 32);
        {
            const int hh = threadIdx.x >> 5, d0 = (threadIdx.x & 31) * 4;
            float* ph = part + hh * nsplit1 * kPartStride;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) {
                const float4 v = *reinterpret_cast<const float4*>(&sO[(w * 4 + hh) * kD + d0]);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            const bool aborted = ctl->abort_flag != 0;
            *reinterpret_cast<float4*>(&ph[4 + d0]) = acc;
            if ((threadIdx.x & 31) == 0) {
                const float mh = (hh == 0) ? M[0] : (hh == 1) ? M[1] : (hh == 2) ? M[2] : M[3];
                ph[0] = aborted ? -INFINITY : mh;
                ph[1] = aborted ? 0.0f : (sL[hh] + sL[4 + hh] + sL[8 + hh] + sL[12 + hh]);
            }
        }
        return;
    }
    // producer warp: meet the consumers at (A), then drain copies that an
    // aborted run left in flight before the CTA's shared memory is released.
    __syncthreads();
    if (lane == 0 && ctl->abort_flag) {
        int done = n;
        for (int w = 0; w < kConsumers; ++w) done = min(done, ctl->consumed[w]);
        for (int kk = done; kk < ctl->issued; ++kk)
            (void)mbar_wait_bounded(smem_u32(&ctl->full[kk % kStages]), (kk / kStages) & 1, kWaitLimitNs, nullptr);
    }
}

// ----------------------------------------------------------------- combine --

__global__ void __launch_bounds__(128) combine_kernel(const DecodeArgs a) {
    const int j = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    const int nsplit1 = a.nsplit + 1;
    const float* parts = a.ws + (size_t)(b * a.hq + j) * nsplit1 * kPartStride;
    float M = -INFINITY;
    for (int s = 0; s < nsplit1; ++s)
        if (parts[s * kPartStride + 1] > 0.0f) M = fmaxf(M, parts[s * kPartStride]);
    float num = 0.0f, den = 0.0f;
    if (M != -INFINITY) {
        for (int s = 0; s < nsplit1; ++s) {
            const float* p = parts + s * kPartStride;
            if (!(p[1] > 0.0f)) continue;
            const float w = ex2(p[0] - M);
            den = fmaf(w, p[1], den);
            num = fmaf(w, p[4 + d], num);
        }
    }
    a.out[((size_t)b * a.hq + j) * kD + d] = (den > 0.0f) ? num / den : 0.0f;
}

// ------------------------------------------------------ bounded-wait test --

__global__ void bounded_wait_kernel(int* err, uint64_t limit_ns) {
    __shared__ unsigned long long bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing ever arrives on this barrier: the wait must give up
        if (!mbar_wait_bounded(smem_u32(&bar), 0, limit_ns, nullptr)) record_error(err, BD_ERR_TIMEOUT);
    }
}

}  // namespace

void decode_splits(int B, int hkv, int max_blocks, int* nsplit, int* pages_per_split) {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            sms = 148;
    }
    const int slots = 2 * sms;
    const int units = max(1, B * hkv);
    int ns = (slots + units - 1) / units;
    ns = max(1, min(ns, max(1, max_blocks)));
    int pps = max(1, (max_blocks + ns - 1) / ns);
    ns = max(1, (max_blocks + pps - 1) / pps);
    *nsplit = ns;
    *pages_per_split = pps;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    static bool attr_set[2] = {false, false};
    const int f = a.format;
    auto kern = (f == BD_FORMAT_NVFP4) ? decode_kernel<BD_FORMAT_NVFP4> : decode_kernel<BD_FORMAT_MXFP4>;
    if (!attr_set[f]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[f] = true;
    }
    dim3 grid((unsigned)(a.nsplit + 1), (unsigned)a.hkv, (unsigned)a.B);
    kern<<<grid, kThreads, kSmemBytes, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    combine_kernel<<<dim3((unsigned)a.hq, (unsigned)a.B), kD, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t s) {
    bounded_wait_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace bd
