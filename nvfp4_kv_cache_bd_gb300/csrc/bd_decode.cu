// Paged single-token decode attention over the hybrid cache (BF16 sink +
// packed FP4 pages + BF16 tail): flash-decoding split-K over pages, then a
// separate kernel that merges the splits.
//
// Method: "How openbitsys/bitdecoding-fp4 works" (decode interface -> paged
// attention kernel; hybrid cache); BitDecoding-FP4 evaluation config
// (config.py): KV_MODES sink_tokens 16, PARITY_ENGINE_KWARGS block_size 128,
// probability_environment ("amax6" / "amax2_or_amax6" with c in {1, 8} and
// tau in [0, 448]), RECIPE dual_residual_query_quantization (two query terms).
//
// Grid (nsplit + 1, kv heads, sequences) of 256-thread CTAs, two per SM.
// Split 0 of a (sequence, kv head) attends the BF16 sink and tail tokens with
// exact probabilities; split s >= 1 takes that sequence's FP4 pages
// [(s - 1) * pages_per_split, s * pages_per_split).  The split-0 CTAs are
// short: the SM slots they free early in a layer let the split combine and
// the next layer's query and decode kernels become resident before this
// decode ends, so the next decode's producers fill their rings during this
// one's tail.
//
// FP4 split CTA: warps 6 and 7 are producers.  One lane of each streams the
// pages' K records (warp 6) or V records (warp 7), in page order, into its
// own 6-slot shared-memory ring with cp.async.bulk (TMA, L2 evict-first),
// completing on per-slot "full" mbarriers; each slot carries the index of
// the page it holds, so a consumer never mistakes an older fill for its own.
// Warps 0..5 consume: each takes the next page from a shared counter, so
// every warp's pages increase and a page's softmax maximum never crosses
// warps.  Per page a warp carries eight 16-token blocks through
//  QK  : m16n8k16 f16 MMAs, M = 16 tokens, N = 8 = 4 query heads x 2 query
//        terms, K = 16 head dims.  FP4 codes are widened by cvt e2m1x2->f16x2
//        and multiplied by their E4M3 scale in f16, which is exact
//        (E2M1 x E4M3 has at most 6 significant bits and lies in
//        [2^-10, 2688]); the query terms are exact the same way.  Per-tensor
//        scales, the 1/sqrt(128) softmax scale and q.mu are applied to the
//        fp32 accumulators.  The K slot is released right after.
//  P   : the page maximum m_p of every head (warp shuffles); P = exp(s - m_p);
//        each 16-token block is quantized to FP4 with the amax2-or-amax6 rule;
//        Phat = E2M1 x E4M3 / c is again exact in f16.  All of this happens
//        before the page's V record is awaited.
//  PV  : O^T[128 dims][8] += Vhat^T[dims][16 tokens] Phat^T.  The V record
//        stores tokens tau and tau+8 in one byte, which is exactly an
//        A-fragment register of this MMA; Phat reaches the B-fragment layout
//        with two warp shuffles.
//  Each warp merges its pages into a running (M, L, O); at the end the
//  consumer warps' states are merged through shared memory into the split
//  partial.
// combine_kernel, one CTA per (sequence, query head), merges the splits:
// O = sum 2^(m-M) O / sum 2^(m-M) l.
//
// The query, decode and combine kernels use programmatic dependent launch:
// the producers start streaming pages while the query quantizer still runs;
// every thread that reads the packed or raw query or the sink/tail rows, or
// writes the workspace or out, first waits on the preceding grid.
#include <math.h>

#include <mutex>

#include "bd_device.cuh"

namespace bd {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kConsumers = 6;                    // consumer warps; warps 6 and 7 stream K and V
constexpr int kThreads = (kConsumers + 2) * 32;
constexpr int kMaxRec = 9216;                    // one K or V record (NVFP4; MXFP4 is 8704 B)
constexpr int kNK = 6, kNV = 6;                  // K-ring and V-ring slots of kMaxRec bytes
constexpr int kRingBytes = (kNK + kNV) * kMaxRec;
constexpr int kWavePages = 32;   // one-wave splits up to this many pages ...
constexpr int kBatchPages = 16;  // ... else splits of this many (more if kMaxSplits needs it)
constexpr int kMaxSplits = 43;    // splits + 1 per (sequence, kv head); the combine stages them in 22.7 KB
constexpr float kSmLog2e = 0.08838834764831845f * 1.4426950408889634f;  // log2(e)/sqrt(128)

struct alignas(16) Ctl {
    unsigned long long fullK[kNK], emptyK[kNK];   // K ring
    unsigned long long fullV[kNV], emptyV[kNV];   // V ring
    float wm[kConsumers + 1][4];   // per-warp running max per head (log2 units); last: BF16 tokens
    float wl[kConsumers + 1][4];   // per-warp softmax denominator per head
    int abort_flag;
    int next_page;             // next page index a consumer warp takes
    int tagK[kNK], tagV[kNV];  // page index each slot's latest fill holds (-1: none)
    int badK[kNK];             // 1: that fill's block-table entry was out of range (no data, skip the page)
};
constexpr int kPTabBytes = 2 * 128 * 4;                        // scale tables (see decode_kernel)
constexpr int kSmemBytes = kRingBytes + (int)sizeof(Ctl) + kPTabBytes;
// Merge area in the (drained) ring: the O of each consumer warp and of the
// BF16 tokens, [kConsumers + 1][4 heads][128] floats; the BF16 staging follows.
constexpr int kStateBytes = (kConsumers + 1) * 4 * 128 * 4;
static_assert(kStateBytes + 2 * 143 * 272 + (4 * 128 + 4 * 144 + 8) * 4 <= kRingBytes,
              "states and sink/tail staging must fit the ring");
static_assert(sizeof(Ctl) % 16 == 0, "the tables after Ctl must stay 16-byte aligned");
static_assert(kMaxSplits <= 64, "the combine handles two splits per lane");

__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// 16-byte asynchronous global -> shared copy (both addresses 16-byte aligned).

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

__device__ __forceinline__ int ld_acquire_shared(const int* p) {
    int v;
    asm volatile("ld.acquire.cta.shared.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_shared(int* p, int v) {
    asm volatile("st.release.cta.shared.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// Wait until the stage holds page `page` and its full barrier has completed
// the phase of the given parity (bounded like mbar_wait_bounded).  The tag is
// read first: the producer publishes it only after the stage's previous fill
// completed and was released, so once the tag matches, the parity test can
// no longer confuse the awaited phase with the one two fills earlier.
__device__ __forceinline__ bool wait_stage_page(uint32_t bar, uint32_t parity, const int* tag, int page,
                                                const volatile int* abort_flag) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (ld_acquire_shared(tag) == page && mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u) {
            if (abort_flag && *abort_flag) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kWaitLimitNs) return false;
        }
    }
}

// Element-wise maximum of v[0..7] over the 8 lanes that share lane & 3 (lane
// bits 2..4), left in every one of them: a reduce-scatter (4 + 2 + 1
// shuffles) leaves each lane the full maximum of one element, an all-gather
// (1 + 2 + 4) returns all eight.  14 shuffles instead of 3 per element.
__device__ __forceinline__ void max8_across_g(float* v, int lane) {
    const bool b2 = lane & 16, b1 = lane & 8, b0 = lane & 4;
    float h4[4];   // elements (b2 ? 4 : 0) + 0..3
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float send = b2 ? v[j] : v[j + 4], keep = b2 ? v[j + 4] : v[j];
        h4[j] = fmaxf(keep, __shfl_xor_sync(kFull, send, 16));
    }
    float h2[2];   // elements (b2 ? 4 : 0) + (b1 ? 2 : 0) + 0..1
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float send = b1 ? h4[j] : h4[j + 2], keep = b1 ? h4[j + 2] : h4[j];
        h2[j] = fmaxf(keep, __shfl_xor_sync(kFull, send, 8));
    }
    // element (b2 ? 4 : 0) + (b1 ? 2 : 0) + (b0 ? 1 : 0), now over all 8 lanes
    const float h1 = fmaxf(b0 ? h2[1] : h2[0], __shfl_xor_sync(kFull, b0 ? h2[0] : h2[1], 4));
    const float o1 = __shfl_xor_sync(kFull, h1, 4);
    const float g2[2] = {b0 ? o1 : h1, b0 ? h1 : o1};
    const float o2[2] = {__shfl_xor_sync(kFull, g2[0], 8), __shfl_xor_sync(kFull, g2[1], 8)};
    const float g4[4] = {b1 ? o2[0] : g2[0], b1 ? o2[1] : g2[1], b1 ? g2[0] : o2[0], b1 ? g2[1] : o2[1]};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float o4 = __shfl_xor_sync(kFull, g4[j], 16);
        v[j] = b2 ? o4 : g4[j];
        v[j + 4] = b2 ? g4[j] : o4;
    }
}

// ------------------------------------------------------ BF16 sink + tail --

// Shared-memory row pitch of a staged bf16 head vector: 256 B plus 16 B so
// that eight consecutive rows read with 16-byte loads hit distinct banks.
constexpr int kRowPitch = 272;
constexpr int kMaxBf16Tok = kSink + kPage - 1;   // 143

// Attention of the 4 query heads of kv head h over the BF16 sink and tail
// tokens of sequence b, left as state slot kConsumers of the CTA merge: O in
// the merge area, the maximum and denominator in ctl (maximum -inf: no
// tokens).  Runs on the whole CTA once the ring is no longer in use.
__device__ void bf16_segment(const DecodeArgs& a, int b, int h, int L, uint8_t* smem, Ctl* ctl) {
    const int ns = min(L, kSink);
    const int rest = max(0, L - kSink);
    const int npages = rest / kPage;
    const int nt = rest - npages * kPage;
    const int T = ns + nt;
    const int tid = threadIdx.x;
    // the sink/tail rows and q may be produced by the preceding grid
    griddep_wait();
    if (T <= 0) {
        if (tid < 4) {
            ctl->wm[kConsumers][tid] = -INFINITY;
            ctl->wl[kConsumers][tid] = 0.0f;
        }
        return;
    }
    float* so = reinterpret_cast<float*>(smem) + kConsumers * 4 * kD;   // this state's O
    uint8_t* ks = smem + kStateBytes;                              // [T][272 B] bf16 keys
    uint8_t* vs = ks + kMaxBf16Tok * kRowPitch;                    // [T][272 B] bf16 values
    float* qf = reinterpret_cast<float*>(vs + kMaxBf16Tok * kRowPitch);   // [4][128]
    float* sp = qf + 4 * kD;                                       // [4][144] scores, then P
    // stage the sink and tail rows of this kv head with asynchronous 16-byte
    // copies (no thread waits for one load before issuing the next)
    for (int i = tid; i < T * 16; i += blockDim.x) {
        const int tau = i >> 4, c = i & 15;
        const size_t krow = tau < ns ? (((size_t)b * kSink + tau) * a.hkv + h) * kD
                                     : (((size_t)b * kPage + (tau - ns)) * a.hkv + h) * kD;
        const uint16_t* kb = (tau < ns ? a.sink_k : a.tail_k) + krow + 8 * c;
        const uint16_t* vb = (tau < ns ? a.sink_v : a.tail_v) + krow + 8 * c;
        cp_async16(smem_u32(ks + tau * kRowPitch + 16 * c), kb);
        cp_async16(smem_u32(vs + tau * kRowPitch + 16 * c), vb);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (tid < 4 * kD / 8) {
        const int hh = tid >> 4, c = tid & 15;
        const uint4 u = *reinterpret_cast<const uint4*>(a.q + ((size_t)b * a.hq + 4 * h + hh) * kD + 8 * c);
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            qf[hh * kD + 8 * c + 2 * e] = bf16_lo(wd[e]);
            qf[hh * kD + 8 * c + 2 * e + 1] = bf16_hi(wd[e]);
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    // scores: two threads per token, four heads.  Thread half hf takes the
    // 16-byte chunks 4hf..4hf+3 and 8+4hf..8+4hf+3 of the row, so the eight
    // lanes of a quarter warp (four tokens, both halves) read distinct banks.
    // The loop bound is the same for the whole CTA (every lane reaches the
    // pair shuffle); a thread past the last token reads row T-1 and stores
    // nothing.
    {
        const int hf = tid & 1;
        for (int base = 0; base < T; base += blockDim.x >> 1) {
            const int tau = base + (tid >> 1);
            const int row = min(tau, T - 1);
            float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const int c = (cc & 3) + 4 * hf + 8 * (cc >> 2);
                const uint4 u = *reinterpret_cast<const uint4*>(ks + row * kRowPitch + 16 * c);
                const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float k0 = bf16_lo(wd[e]), k1 = bf16_hi(wd[e]);
                    const int d = 8 * c + 2 * e;
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {
                        const float2 qq = *reinterpret_cast<const float2*>(&qf[hh * kD + d]);
                        s[hh] = fmaf(qq.y, k1, fmaf(qq.x, k0, s[hh]));
                    }
                }
            }
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) s[hh] += __shfl_xor_sync(kFull, s[hh], 1);
            if (hf == 0 && tau < T) {
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) sp[hh * 144 + tau] = s[hh] * kSmLog2e;
            }
        }
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
            ctl->wm[kConsumers][warp] = m;
            ctl->wl[kConsumers][warp] = l;
        }
    }
    __syncthreads();
    // O = P V: thread (head dim d, head pair hp), all 256 threads
    {
        const int d = tid & (kD - 1), hp = tid >> 7;
        const float* p0 = sp + (2 * hp) * 144;
        const float* p1 = p0 + 144;
        float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll 4
        for (int tau = 0; tau < T; ++tau) {
            const float v = __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(vs + tau * kRowPitch + 2 * d)) << 16);
            acc0 = fmaf(p0[tau], v, acc0);
            acc1 = fmaf(p1[tau], v, acc1);
        }
        so[(2 * hp) * kD + d] = acc0;
        so[(2 * hp + 1) * kD + d] = acc1;
    }
}

// ------------------------------------------------ FP4 page split: consumer --

template <int FMT, int PM>
__device__ void consume_pages(const DecodeArgs& a, int b, int h, int n, uint8_t* smem, Ctl* ctl, int warp,
                              int lane) {
    const int g = lane >> 2, t = lane & 3;
    griddep_wait();
    const uint8_t* qrec = a.qp + (size_t)b * a.qstride;
    const int hq = a.hq;
    // B fragments of the query: row n = g -> head 4h + g/2, term g%2; this
    // lane's k-slots are head dims 32t .. 32t+31.
    uint32_t qB[16];
    float qx[2];   // MXFP4: 2^(reference exponent) of this lane's two C columns
    {
        const int jq = 4 * h + (g >> 1), term = g & 1;
        const uint4 qc = *reinterpret_cast<const uint4*>(qrec + (term * hq + jq) * 64 + 16 * t);
        uint32_t slo, shi;
        if (FMT == BD_FORMAT_NVFP4) {
            const uint32_t qsd = e4m3x2_to_f16x2(
                *reinterpret_cast<const uint16_t*>(qrec + 2 * hq * 64 + (term * hq + jq) * 8 + 2 * t));
            slo = bcast_lo(qsd);
            shi = bcast_hi(qsd);
        } else {
            const uint32_t e4 = *reinterpret_cast<const uint32_t*>(qrec + 2 * hq * 64 + (term * hq + jq) * 4);
            int emax = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) emax = max(emax, (int)((e4 >> (8 * q)) & 0xFF));
            slo = shi = bcast_lo(f16_pow2((int)((e4 >> (8 * t)) & 0xFF) - emax));
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t pr = byte_pair(qc, kk);
            const uint32_t sc = kk < 4 ? slo : shi;
            qB[2 * kk] = hmul2(e2m1x2_to_f16x2(pr & 0xFF), sc);
            qB[2 * kk + 1] = hmul2(e2m1x2_to_f16x2(pr >> 8), sc);
        }
        qx[0] = qx[1] = 1.0f;
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
        }
    }
    const float* gq = reinterpret_cast<const float*>(qrec + 2 * hq * 64 + 2 * hq * 8);
    const float gK = (FMT == BD_FORMAT_NVFP4) ? a.gk : 1.0f;
    const float gV = (FMT == BD_FORMAT_NVFP4) ? a.gv : 1.0f;
    const float a1 = kSmLog2e * gK * ((FMT == BD_FORMAT_NVFP4) ? gq[0] : qx[0]);
    const float a2 = kSmLog2e * gK * ((FMT == BD_FORMAT_NVFP4) ? gq[1] : qx[1]);
    const float bq = a.centering ? kSmLog2e * gq[4 + 4 * h + t] : 0.0f;
    const float ccf = (float)((PM == BD_P_AMAX2_OR_AMAX6) ? a.p_c : 1);
    const float tau = a.tau;
    // per-byte tables (see decode_kernel): [0,128) 1/sd, [128,256) (sd/c, sd/c)
    // f16x2
    const float* ptab_rcp = reinterpret_cast<const float*>(smem + kRingBytes + sizeof(Ctl));
    const uint32_t* ptab_sdc = reinterpret_cast<const uint32_t*>(ptab_rcp + 128);
    const int srcA = (lane & ~3) | ((2 * t) & 3), srcB = (lane & ~3) | ((2 * t + 1) & 3);
    const int gs = g & 3;

    float Mt = -INFINITY, MA = -INFINITY, MB = -INFINITY;   // running max of heads t, 2t, 2t+1
    float lacc = 0.0f;
    float o[8][4];
#pragma unroll
    for (int bm = 0; bm < 8; ++bm) o[bm][0] = o[bm][1] = o[bm][2] = o[bm][3] = 0.0f;

    for (;;) {
        // the next page in order: warps take pages as they become free, so
        // every warp's pages increase and the lowest unfinished page can
        // always proceed
        int k = 0;
        if (lane == 0) k = atomicAdd(&ctl->next_page, 1);
        k = __shfl_sync(kFull, k, 0);
        if (k >= n) break;
        const int sk = k % kNK, sv = k % kNV;
        // A warp may start waiting for fill j of a slot before fill j-1 has
        // landed; the phase parity alone cannot tell fill j-2 from fill j, the
        // page tag can.
        if (!wait_stage_page(smem_u32(&ctl->fullK[sk]), (k / kNK) & 1, &ctl->tagK[sk], k, &ctl->abort_flag)) {
            if (!ctl->abort_flag) record_error(a.err, BD_ERR_TIMEOUT);
            ctl->abort_flag = 1;
            break;
        }
        if (ctl->badK[sk]) {
            // out-of-range block-table entry: nothing was copied for this page
            // and it is left out; hand both slots back in ring order
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->emptyK[sk]));
            if (!wait_stage_page(smem_u32(&ctl->fullV[sv]), (k / kNV) & 1, &ctl->tagV[sv], k, &ctl->abort_flag)) {
                if (!ctl->abort_flag) record_error(a.err, BD_ERR_TIMEOUT);
                ctl->abort_flag = 1;
                break;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->emptyV[sv]));
            continue;
        }
        const uint8_t* Ks = smem + sk * kMaxRec;
        const uint8_t* Vs = smem + (kNK + sv) * kMaxRec;

        // ---------------- QK over the eight 16-token blocks: log2-scaled
        // scores of head t for tokens 16mi+g and 16mi+g+8 stay in registers
        float sc[16];
        float mp = -INFINITY;
#pragma unroll
        for (int mi = 0; mi < 8; ++mi) {
            {
                const int tok0 = 16 * mi + g, tok1 = tok0 + 8;
                const uint4 c0 = lds128(Ks + tok0 * 64 + 16 * t);
                const uint4 c1 = lds128(Ks + tok1 * 64 + 16 * t);
                uint32_t s0lo, s0hi, s1lo, s1hi;
                float fk0 = 1.0f, fk1 = 1.0f;
                if (FMT == BD_FORMAT_NVFP4) {
                    // scale bytes of blocks 2t, 2t+1 of both rows, one 16-bit
                    // load per row, widened exactly to f16 and broadcast to
                    // (sd, sd) pairs
                    const uint32_t h0 = e4m3x2_to_f16x2(lds16(Ks + kCodeBytes + tok0 * 8 + 2 * t));
                    const uint32_t h1 = e4m3x2_to_f16x2(lds16(Ks + kCodeBytes + tok1 * 8 + 2 * t));
                    s0lo = bcast_lo(h0);
                    s0hi = bcast_hi(h0);
                    s1lo = bcast_lo(h1);
                    s1hi = bcast_hi(h1);
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
                // two accumulators halve the dependent MMA chain of the block
                float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t cw0[4] = {c0.x, c0.y, c0.z, c0.w}, cw1[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // word j holds bytes 4j..4j+3: k-tiles 2j (bytes 4j, 4j+1) and 2j+1
                    uint32_t f0[4], f1[4];
                    e2m1x8_to_f16x2x4(cw0[j], f0);
                    e2m1x8_to_f16x2x4(cw1[j], f1);
                    const uint32_t sa = j < 2 ? s0lo : s0hi, sb2 = j < 2 ? s1lo : s1hi;
                    uint32_t A[4];
                    A[0] = hmul2(f0[0], sa);
                    A[1] = hmul2(f1[0], sb2);
                    A[2] = hmul2(f0[1], sa);
                    A[3] = hmul2(f1[1], sb2);
                    mma16816(acc, A, qB[4 * j], qB[4 * j + 1]);
                    A[0] = hmul2(f0[2], sa);
                    A[1] = hmul2(f1[2], sb2);
                    A[2] = hmul2(f0[3], sa);
                    A[3] = hmul2(f1[3], sb2);
                    mma16816(acc2, A, qB[4 * j + 2], qB[4 * j + 3]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] += acc2[e];
                const float s0 = fmaf(fk0, fmaf(acc[1], a2, acc[0] * a1), bq);
                const float s1 = fmaf(fk1, fmaf(acc[3], a2, acc[2] * a1), bq);
                sc[2 * mi] = s0;
                sc[2 * mi + 1] = s1;
                mp = fmaxf(mp, fmaxf(s0, s1));
            }
        }

        // the K slot is free once every lane's key reads are done
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->emptyK[sk]));

        // ---------------- page maximum of head t (and of heads 2t, 2t+1)
        mp = fmaxf(mp, __shfl_xor_sync(kFull, mp, 4));
        mp = fmaxf(mp, __shfl_xor_sync(kFull, mp, 8));
        mp = fmaxf(mp, __shfl_xor_sync(kFull, mp, 16));
        const float mpA = __shfl_sync(kFull, mp, srcA), mpB = __shfl_sync(kFull, mp, srcB);

        // ---------------- per 16-token block: probabilities and their FP4
        // quantization into P V's B fragments, all before the page's V record
        // is awaited (its slot is held only for P V).  NVFP4: the running max
        // is updated first and
        // the page weight 2^(m_p - M) is folded into the f16 Phat operand, so
        // P V accumulates straight into O (one f16 rounding, < 2^-11
        // relative, per weighted Phat).  MXFP4 keeps a per-page O_p because
        // its V reference exponent changes from page to page.
        const float mnt = fmaxf(Mt, mp);
        const float wpage = ex2(mp - mnt);
        uint32_t wh = 0x3C003C00u;   // (1, 1)
        float op[8][4];
        if (FMT == BD_FORMAT_NVFP4) {
            const float mnA = fmaxf(MA, mpA), mnB = fmaxf(MB, mpB);
            const float aA = ex2(MA - mnA), aB = ex2(MB - mnB);
            if (__any_sync(kFull, (aA != 1.0f) | (aB != 1.0f))) {
#pragma unroll
                for (int bm = 0; bm < 8; ++bm) {
                    o[bm][0] *= aA;
                    o[bm][1] *= aB;
                    o[bm][2] *= aA;
                    o[bm][3] *= aB;
                }
            }
            MA = mnA;
            MB = mnB;
            wh = bcast_lo((uint32_t)__half_as_ushort(__float2half_rn(wpage)));
        } else {
#pragma unroll
            for (int bm = 0; bm < 8; ++bm) op[bm][0] = op[bm][1] = op[bm][2] = op[bm][3] = 0.0f;
        }
        // the page's probabilities first, then the eight blocks' maxima of
        // u = c P over their 16 tokens with one reduction across the lanes g
        float pr[16];
        float lpage = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            pr[2 * i] = ex2(sc[2 * i] - mp);
            pr[2 * i + 1] = ex2(sc[2 * i + 1] - mp);
            lpage += pr[2 * i] + pr[2 * i + 1];
        }
        float bmax[8];
        uint32_t bfr[16];   // B fragments of Phat for P V, two per block
        if (PM != BD_P_NONE) {
#pragma unroll
            for (int i = 0; i < 8; ++i) bmax[i] = fmaxf(pr[2 * i] * ccf, pr[2 * i + 1] * ccf);
            max8_across_g(bmax, lane);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            {
                const float p0 = pr[2 * i], p1 = pr[2 * i + 1];
                uint32_t pv;
                if (PM == BD_P_NONE) {
                    const __half2 hh = __floats2half2_rn(p0, p1);
                    pv = *reinterpret_cast<const uint32_t*>(&hh);
                } else {
                    const float u0 = p0 * ccf, u1 = p1 * ccf;
                    const float am = bmax[i];
                    const bool two = (PM == BD_P_AMAX2_OR_AMAX6) && (am < tau);
                    const float sv = two ? am * 0.5f : div6(am);
                    // scale byte -> 1/sd (correctly rounded) and (sd/c, sd/c) from the tables;
                    // byte 0 is the zero scale (S == 0: all codes zero)
                    const uint32_t sbyte = e4m3(sv);
                    const float inv = ptab_rcp[sbyte];
                    const uint32_t byte = (sbyte == 0) ? 0u : e2m1x2(__fmul_rn(u0, inv), __fmul_rn(u1, inv));
                    pv = hmul2(e2m1x2_to_f16x2(byte), ptab_sdc[sbyte]);
                }
                if (FMT == BD_FORMAT_NVFP4) pv = hmul2(pv, wh);
                // lanes with g >= 4 feed the padding columns 4..7 (duplicates of
                // heads 0..3); their outputs are never read
                bfr[2 * i] = __shfl_sync(kFull, pv, 4 * t + gs);
                bfr[2 * i + 1] = __shfl_sync(kFull, pv, 16 + 4 * t + gs);
            }
        }

        // ---------------- P V: only now is the page's V record needed
        if (!wait_stage_page(smem_u32(&ctl->fullV[sv]), (k / kNV) & 1, &ctl->tagV[sv], k, &ctl->abort_flag)) {
            if (!ctl->abort_flag) record_error(a.err, BD_ERR_TIMEOUT);
            ctl->abort_flag = 1;
            break;
        }

        float fv = 1.0f;   // MXFP4: 2^(reference exponent of this lane's V block)
        int ev_ref = 0;
        if (FMT == BD_FORMAT_MXFP4) {
            int em = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
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
        for (int i = 0; i < 8; ++i) {
            {
                const uint32_t b01 = bfr[2 * i], b23 = bfr[2 * i + 1];
                // dims 16g .. 16g+15 of pair rows t and t+4 sit at slot
                // g ^ 2t: each quarter warp's eight 16-byte reads cover all
                // 32 banks
                const uint4 v0 = lds128(Vs + (i * 8 + t) * kD + 16 * (g ^ (2 * t)));
                const uint4 v1 = lds128(Vs + (i * 8 + t + 4) * kD + 16 * (g ^ (2 * t)));
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
                const uint32_t vw0[4] = {v0.x, v0.y, v0.z, v0.w}, vw1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // word j holds dims 16g+4j .. 16g+4j+3: m-tiles 2j (dims 4j, 4j+1) and 2j+1
                    uint32_t f0[4], f1[4];
                    e2m1x8_to_f16x2x4(vw0[j], f0);
                    e2m1x8_to_f16x2x4(vw1[j], f1);
                    uint32_t A[4];
                    A[0] = hmul2(f0[0], vs0);
                    A[1] = hmul2(f0[1], vs0);
                    A[2] = hmul2(f1[0], vs1);
                    A[3] = hmul2(f1[1], vs1);
                    mma16816(FMT == BD_FORMAT_NVFP4 ? o[2 * j] : op[2 * j], A, b01, b23);
                    A[0] = hmul2(f0[2], vs0);
                    A[1] = hmul2(f0[3], vs0);
                    A[2] = hmul2(f1[2], vs1);
                    A[3] = hmul2(f1[3], vs1);
                    mma16816(FMT == BD_FORMAT_NVFP4 ? o[2 * j + 1] : op[2 * j + 1], A, b01, b23);
                }
            }
        }
        // release the V slot: every lane's shared-memory reads are done
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->emptyV[sv]));

        // ---------------- merge the page into the warp's running state
        lacc = fmaf(lacc, ex2(Mt - mnt), wpage * lpage);
        Mt = mnt;
        if (FMT == BD_FORMAT_MXFP4) {
            const float mnA = fmaxf(MA, mpA), mnB = fmaxf(MB, mpB);
            const float aA = ex2(MA - mnA), aB = ex2(MB - mnB);
            const float bA = ex2(mpA - mnA) * fv, bB = ex2(mpB - mnB) * fv;
            MA = mnA;
            MB = mnB;
#pragma unroll
            for (int bm = 0; bm < 8; ++bm) {
                o[bm][0] = fmaf(o[bm][0], aA, bA * op[bm][0]);
                o[bm][1] = fmaf(o[bm][1], aB, bB * op[bm][1]);
                o[bm][2] = fmaf(o[bm][2], aA, bA * op[bm][2]);
                o[bm][3] = fmaf(o[bm][3], aB, bB * op[bm][3]);
            }
        }
    }

    // ---------------- hand the warp state to the CTA merge
    __syncthreads();   // (A) all consumers are done with the ring
    float* sO = reinterpret_cast<float*>(smem);   // [consumer warps][4 heads][128]
    if (t < 2) {
#pragma unroll
        for (int bm = 0; bm < 8; ++bm) {
            const int d = 16 * g + 2 * bm;
            sO[(warp * 4 + 2 * t) * kD + d] = o[bm][0] * gV;
            sO[(warp * 4 + 2 * t + 1) * kD + d] = o[bm][1] * gV;
            sO[(warp * 4 + 2 * t) * kD + d + 1] = o[bm][2] * gV;
            sO[(warp * 4 + 2 * t + 1) * kD + d + 1] = o[bm][3] * gV;
        }
    }
    lacc += __shfl_xor_sync(kFull, lacc, 4);
    lacc += __shfl_xor_sync(kFull, lacc, 8);
    lacc += __shfl_xor_sync(kFull, lacc, 16);
    if (g == 0) {
        ctl->wm[warp][t] = Mt;
        ctl->wl[warp][t] = lacc;
    }
}

// CTA merge of the states (consumer warps, then the BF16 tokens) into this
// split's partial; a state with maximum -inf holds nothing and is skipped.
__device__ void write_split_partial(const DecodeArgs& a, float* part, const uint8_t* smem, const Ctl* ctl) {
    const int tid = threadIdx.x;
    if (tid >= 128) return;
    const int hh = tid >> 5, d0 = (tid & 31) * 4;
    const int nparts = a.nsplit + 1;
    const float* sO = reinterpret_cast<const float*>(smem);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w <= kConsumers; ++w) M = fmaxf(M, ctl->wm[w][hh]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.0f;
#pragma unroll
    for (int w = 0; w <= kConsumers; ++w) {
        if (ctl->wm[w][hh] == -INFINITY) continue;
        const float e = ex2(ctl->wm[w][hh] - M);
        const float4 v = *reinterpret_cast<const float4*>(&sO[(w * 4 + hh) * kD + d0]);
        acc.x = fmaf(e, v.x, acc.x);
        acc.y = fmaf(e, v.y, acc.y);
        acc.z = fmaf(e, v.z, acc.z);
        acc.w = fmaf(e, v.w, acc.w);
        L = fmaf(e, ctl->wl[w][hh], L);
    }
    float* ph = part + hh * nparts * kPartStride;
    *reinterpret_cast<float4*>(&ph[4 + d0]) = acc;
    if ((tid & 31) == 0) {
        const bool aborted = ctl->abort_flag != 0 || M == -INFINITY;
        ph[0] = aborted ? -INFINITY : M;
        ph[1] = aborted ? 0.0f : L;
    }
}

// Merge the split partials of (sequence b, query head j) into out: one CTA
// of 128 threads per (b, j), launched after the decode with programmatic
// dependent launch.  The head's partials (one contiguous block of
// nsplit + 1 records) are staged into shared memory with 16-byte
// asynchronous copies; warp 0 finds the maximum M over the splits (one
// integer warp reduction of order-preserving keys), the weights
// w_s = 2^(m_s - M) (0 for an empty split) and the denominator sum w_s l_s;
// thread d then sums w_s O_s[d].
__global__ void __launch_bounds__(128) combine_kernel(const DecodeArgs a) {
    __shared__ __align__(16) float sp[kMaxSplits * kPartStride];
    __shared__ float sw[kMaxSplits];
    __shared__ float sden;
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int bj = blockIdx.x;   // b * hq + j
    const int nparts = a.nsplit + 1;   // partials per (sequence, query head)
    const int tid = threadIdx.x, lane = tid & 31;
    const float* base = a.parts + (size_t)bj * nparts * kPartStride;
    griddep_wait();   // the decode grid has completed: its partials are visible
    for (int i = tid; i < nparts * (kPartStride / 4); i += blockDim.x) cp_async16(smem_u32(sp + 4 * i), base + 4 * i);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (tid < 32) {
        float m[2], l[2];
        uint32_t key = 0;   // order-preserving u32 key of the largest m with l > 0
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int sidx = lane + 32 * r;
            m[r] = (sidx < nparts) ? sp[sidx * kPartStride] : -INFINITY;
            l[r] = (sidx < nparts) ? sp[sidx * kPartStride + 1] : 0.0f;
            if (l[r] > 0.0f) key = max(key, f32_order_key(m[r]));
        }
        key = __reduce_max_sync(kFull, key);
        const float M = (key == 0) ? -INFINITY : f32_from_order_key(key);
        float den = 0.0f;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int sidx = lane + 32 * r;
            const float w = (l[r] > 0.0f) ? ex2(m[r] - M) : 0.0f;
            if (sidx < nparts) sw[sidx] = w;
            den = fmaf(w, l[r], den);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
        if (lane == 0) sden = den;
    }
    __syncthreads();
    const float* ph = sp + 4 + tid;
    float n0 = 0.0f, n1 = 0.0f;
    int sidx = 0;
#pragma unroll 4
    // an empty split wrote no O (its workspace bytes may hold anything, NaN
    // included): it is skipped, not multiplied by its zero weight
    for (; sidx + 1 < nparts; sidx += 2) {
        const float w0 = sw[sidx], w1 = sw[sidx + 1];
        if (w0 != 0.0f) n0 = fmaf(w0, ph[sidx * kPartStride], n0);
        if (w1 != 0.0f) n1 = fmaf(w1, ph[(sidx + 1) * kPartStride], n1);
    }
    if (sidx < nparts && sw[sidx] != 0.0f) n0 = fmaf(sw[sidx], ph[sidx * kPartStride], n0);
    const float den = sden;
    a.out[(size_t)bj * kD + tid] = (den > 0.0f) ? (n0 + n1) * (1.0f / den) : 0.0f;
}

template <int FMT, int PM>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const DecodeArgs a) {   // 128 registers
    extern __shared__ __align__(128) uint8_t smem[];
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    // a negative length counts as 0; one past the block table's capacity keeps
    // its first max_blocks pages; both are argument errors
    const int Lraw = a.seq_lens[b];
    const int L = max(0, Lraw);
    if (split == 0 && h == 0 && threadIdx.x == 0 &&
        (Lraw < 0 || (int64_t)Lraw > kSink + (int64_t)kPage * a.max_blocks + (kPage - 1)))
        record_error(a.err, BD_ERR_INVALID_ARG);
    float* part = a.parts + ((size_t)(b * a.hq + 4 * h) * (a.nsplit + 1) + split) * kPartStride;
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + kRingBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Let the next kernel in the stream launch now: this kernel reads the
    // query (and its sink/tail rows) and writes the workspace and out only
    // after griddepcontrol.wait, so its producers can start streaming the
    // layer's static FP4 pages while the previous grid still drains.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // pages past the block-table row are ignored (the header bounds L)
    const int npages = min(max(0, L - kSink) / kPage, a.max_blocks);
    const bool bf16 = split == 0;   // the BF16 sink and tail tokens, no FP4 pages
    const int p0 = bf16 ? 0 : (split - 1) * a.pages_per_split;
    const int p1 = bf16 ? 0 : min(p0 + a.pages_per_split, npages);

    if (p0 >= p1 && !bf16) {
        griddep_wait();
        if (threadIdx.x < 4) {
            part[threadIdx.x * (a.nsplit + 1) * kPartStride + 0] = -INFINITY;
            part[threadIdx.x * (a.nsplit + 1) * kPartStride + 1] = 0.0f;
        }
        return;
    }
    if (p0 >= p1) {
        // no FP4 pages: the consumer states are empty and nothing aborted
        if (threadIdx.x < kConsumers * 4) {
            ctl->wm[threadIdx.x >> 2][threadIdx.x & 3] = -INFINITY;
            ctl->wl[threadIdx.x >> 2][threadIdx.x & 3] = 0.0f;
        }
        if (threadIdx.x == 0) ctl->abort_flag = 0;
    } else {
        const int n = p1 - p0;
        constexpr int RB = (FMT == BD_FORMAT_NVFP4) ? 9216 : 8704;
        if (threadIdx.x == 0) {
            for (int s = 0; s < kNK; ++s) {
                mbar_init(smem_u32(&ctl->fullK[s]), 1);
                mbar_init(smem_u32(&ctl->emptyK[s]), 1);
                ctl->tagK[s] = -1;
                ctl->badK[s] = 0;
            }
            for (int s = 0; s < kNV; ++s) {
                mbar_init(smem_u32(&ctl->fullV[s]), 1);
                mbar_init(smem_u32(&ctl->emptyV[s]), 1);
                ctl->tagV[s] = -1;
            }
            ctl->abort_flag = 0;
            ctl->next_page = 0;
            fence_mbar_init();
        }
        if (threadIdx.x < 128) {
            // exact per-byte tables for the E4M3 scale byte bb: the correctly
            // rounded 1/sd and the f16x2 pair (sd/c, sd/c) for the probability
            // quantizer (exact: c is a power of two)
            float* tab = reinterpret_cast<float*>(smem + kRingBytes + sizeof(Ctl));
            const uint32_t bb = threadIdx.x;
            const float sd = e4m3_value(bb);
            const float cc = (float)((PM == BD_P_AMAX2_OR_AMAX6) ? a.p_c : 1);
            tab[bb] = (bb == 0) ? 0.0f : __frcp_rn(sd);
            const uint32_t sdh = e4m3x2_to_f16x2(bb);
            const uint32_t icc = bcast_lo((uint32_t)__half_as_ushort(__float2half_rn(1.0f / cc)));
            reinterpret_cast<uint32_t*>(tab)[128 + bb] = hmul2(bcast_lo(sdh), icc);
        }
        __syncthreads();
        if (warp >= kConsumers) {
            // --------------------------------------------------- producers --
            // warp 6 streams the pages' K records into the K ring, warp 7 their
            // V records into the V ring, each in page order
            const bool isK = (warp == kConsumers);
            const int N = isK ? kNK : kNV;
            unsigned long long* fullb = isK ? ctl->fullK : ctl->fullV;
            unsigned long long* emptyb = isK ? ctl->emptyK : ctl->emptyV;
            int* tag = isK ? ctl->tagK : ctl->tagV;
            uint8_t* slots = smem + (isK ? 0 : kNK * kMaxRec);
            if (lane == 0) {
                const int32_t* bt = a.block_table + (size_t)b * a.max_blocks + p0;
                // each page is read once per call: evict it from L2 first
                const uint64_t policy = l2_evict_first_policy();
                for (int k = 0; k < n; ++k) {
                    const int s = k % N;
                    if (k >= N && !mbar_wait_bounded(smem_u32(&emptyb[s]), ((k / N) - 1) & 1, kWaitLimitNs,
                                                     &ctl->abort_flag)) {
                        if (!ctl->abort_flag) record_error(a.err, BD_ERR_TIMEOUT);
                        ctl->abort_flag = 1;
                        break;
                    }
                    const int64_t phys = bt[k];
                    const bool ok = page_ok(phys, a.pool_pages);
                    const uint32_t full = smem_u32(&fullb[s]);
                    if (isK) ctl->badK[s] = ok ? 0 : 1;   // published by the tag's release
                    // tag the fill before it is armed: consumers accept a completed
                    // phase only together with their own page index
                    st_release_shared(&tag[s], k);
                    if (ok) {
                        const uint8_t* rec = a.pool + ((phys * a.hkv + h) * 2 + (isK ? 0 : 1)) * (int64_t)RB;
                        mbar_arrive_expect_tx(full, RB);
                        bulk_g2s_hint(smem_u32(slots + s * kMaxRec), rec, RB, full, policy);
                    } else {
                        // an entry outside the pool: complete the phase without data
                        if (isK) record_error(a.err, BD_ERR_INVALID_ARG);
                        mbar_arrive(full);
                    }
                }
            }
            __syncthreads();   // (A)
            // an aborted run drains the copies it left in flight before the ring
            // is reused: a slot's last fill is the only one that can be pending
            if (lane == 0 && ctl->abort_flag) {
                for (int s = 0; s < N; ++s) {
                    const int f = tag[s];
                    if (f >= 0) (void)mbar_wait_bounded(smem_u32(&fullb[s]), (f / N) & 1, kWaitLimitNs, nullptr);
                }
            }
        } else {
            consume_pages<FMT, PM>(a, b, h, n, smem, ctl, warp, lane);   // contains (A)
        }
    }
    if (!bf16 && threadIdx.x < 4) {
        ctl->wm[kConsumers][threadIdx.x] = -INFINITY;
        ctl->wl[kConsumers][threadIdx.x] = 0.0f;
    }
    __syncthreads();   // (B) warp states and drained ring
    if (bf16) bf16_segment(a, b, h, L, smem, ctl);   // the same for the whole CTA
    __syncthreads();
    write_split_partial(a, part, smem, ctl);
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

namespace {

// Host state of the decode launcher per device, filled on first use under one
// lock: the SM count and which decode instances have their dynamic
// shared-memory limit raised (a per-device function attribute).
struct DeviceState {
    int sms = 0;
    bool smem_attr[2][3] = {};
};
std::mutex g_dev_lock;
DeviceState g_dev[kMaxDevices];

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

int device_sms() {
    const int dev = current_device();
    if (dev < 0) return 148;
    std::lock_guard<std::mutex> g(g_dev_lock);
    int& sms = g_dev[dev].sms;
    if (sms <= 0 && (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0))
        sms = 148;
    return sms;
}

}  // namespace

void decode_splits(int B, int hkv, int max_blocks, int* nsplit, int* pages_per_split) {
    const int sms = device_sms();
    // two CTAs fit per SM; split 0 of every (sequence, kv head) is the BF16
    // sink/tail CTA, so a single wave holds units * (splits + 1) CTAs
    const int slots = 2 * sms;
    const int units = max(1, B * hkv);
    int ns = max(1, slots / units - 1);
    ns = max(1, min(ns, max(1, max_blocks)));
    int pps = max(1, (max_blocks + ns - 1) / ns);
    // When one wave would give a split many pages (a batch of long and short
    // sequences: the host does not know the lengths), use short splits
    // instead: a split past its sequence's pages exits at once and the
    // hardware scheduler spreads the rest over several waves.
    if (pps > kWavePages) pps = max(kBatchPages, (max_blocks + kMaxSplits - 2) / (kMaxSplits - 1));
    ns = max(1, (max_blocks + pps - 1) / pps);
    if (ns > kMaxSplits - 1) {
        pps = (max_blocks + kMaxSplits - 2) / (kMaxSplits - 1);
        ns = (max_blocks + pps - 1) / pps;
    }
    *nsplit = ns;
    *pages_per_split = pps;
}

size_t decode_ws_bytes(int B, int hq, int nsplit) {
    return (size_t)B * hq * (nsplit + 1) * kPartStride * sizeof(float);
}

using DecodeFn = void (*)(DecodeArgs);

template <int FMT>
DecodeFn pick_decode(int p_mode) {
    if (p_mode == BD_P_NONE) return decode_kernel<FMT, BD_P_NONE>;
    if (p_mode == BD_P_AMAX6) return decode_kernel<FMT, BD_P_AMAX6>;
    return decode_kernel<FMT, BD_P_AMAX2_OR_AMAX6>;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    const int f = a.format, pm = a.p_mode;
    DecodeFn kern = (f == BD_FORMAT_NVFP4) ? pick_decode<BD_FORMAT_NVFP4>(pm) : pick_decode<BD_FORMAT_MXFP4>(pm);
    {
        const int dev = current_device();
        if (dev < 0) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> g(g_dev_lock);
        if (!g_dev[dev].smem_attr[f][pm]) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess) return e;
            g_dev[dev].smem_attr[f][pm] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.nsplit + 1), (unsigned)a.hkv, (unsigned)a.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return e;
    // the split combine, dependent on the decode grid
    cfg.gridDim = dim3((unsigned)(a.B * a.hq));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

// ------------------------------------------- fixed scratch (no allocation) --
//
// bd_decode_attention_noalloc serves callers that cannot call cudaMalloc --
// for example code running inside another framework's memory pool, a plugin
// that is handed only its input and output buffers, or a process whose GPU
// memory is reserved up front.  Its split partials live in this file-scope
// array instead of a caller workspace (nothing in it has to start at zero).  Every GPU that loads
// the library holds the array until the process exits; every call shares it,
// so calls that overlap on the GPU race.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

cudaError_t noalloc_scratch(void** out) {
    // In host code g_noalloc_scratch names a host-side stand-in, not device
    // memory: the device address is looked up once per device, with that
    // device current, and cached.
    static std::mutex lock;
    static void* addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(lock);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

cudaError_t launch_bounded_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t s) {
    bounded_wait_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace bd
