// Paged single-token decode attention over the hybrid cache (BF16 sink +
// packed FP4 pages + BF16 tail): flash-decoding split-K over pages, the
// splits merged by the last split of each (sequence, kv head) to finish.
//
// Method: "How openbitsys/bitdecoding-fp4 works" (decode interface -> paged
// attention kernel; hybrid cache); BitDecoding-FP4 evaluation config
// (config.py): KV_MODES sink_tokens 16, PARITY_ENGINE_KWARGS block_size 128,
// probability_environment ("amax6" / "amax2_or_amax6" with c in {1, 8} and
// tau in [0, 448]), RECIPE dual_residual_query_quantization (two query terms).
//
// Grid (nsplit + 1, kv heads, sequences) of 256-thread CTAs, two per SM; a
// single-wave grid leaves a few SM slots free, where the next layer's CTAs
// start early.  Split 0 of a (sequence, kv head) attends the BF16 sink and tail
// tokens with exact probabilities; split s >= 1 takes that sequence's FP4
// pages [(s - 1) * pages_per_split, s * pages_per_split).  As this layer's
// CTAs finish, the next layer's decode CTAs take their slots, so the next
// decode's producers load its first round of pages during this one's tail.
//
// FP4 split CTA, two warpgroups with their own register shares:
//  warp 0    streams the pages' K records, in page order, into a 4-slot
//            shared-memory ring with cp.async.bulk (TMA, L2 evict-first);
//  warp 1    streams the V records into a 6-slot V ring the same way;
//  warp 2    computes every page's scores on the tensor core: the block-scaled
//            tcgen05 MMA (kind::mxf4nvf4) takes the K record's FP4 codes
//            (the B operand, N = the page's 128 tokens) and its E4M3 / UE8M0
//            block scales straight from shared memory, the query (A operand,
//            M = 128: 4 heads x 2 terms in lane quarter w, every other row
//            zero) and its scales, and accumulates fp32 scores in tensor
//            memory.  Pages go in rounds of four: page 4 r + w lands in lane
//            quarter w of one 128-column score buffer (the first MMA of a
//            round overwrites the buffer, the rest accumulate, and zero query
//            rows leave the other quarters as they are);
//  warp 3    owns the CTA's 256 TMEM columns (the score buffer, the query's
//            scale factors and three pages' K scale factors);
//  warps 4-7 consume: warp 4 + w takes page 4 r + w of every round alone.
//            One tcgen05 load (16x256b) gives lane (g, t) the scores of query
//            head g (both terms) for tokens 8 j + 2 t, 8 j + 2 t + 1 -- the
//            B-fragment layout of the P V MMA -- so the page maximum is a
//            register reduction plus two shuffles, each 16-token block's FP4
//            probabilities (amax2-or-amax6) are quantized in place, and P V
//            runs as m16n8k16 f16 MMAs (O^T[128 dims][8] += Vhat^T Phat^T; V's
//            scales run along head_dim, the MMA's output dimension, so a
//            block-scaled MMA cannot take V).  Lanes of rows 4..7 carry no
//            query head; their results are never read.
// Every page's K and V record is read once from HBM; each page is processed
// by one warp in a fixed order, so a split's result does not depend on
// scheduling.  Split 0 and every split with pages write their partial (m,
// l, O per query head) to the workspace and count themselves in at their
// (sequence, kv head)'s arrival counter (a split past its sequence's pages
// exits at once; each CTA knows from the length how many splits hold
// pages); the split that completes the count merges that group's partials,
// O = sum 2^(m-M) O / sum 2^(m-M) l, in a fixed split order, so the result
// does not depend on which split came last either.  With no separate merge
// kernel, a layer is one grid: nothing of a layer's chain holds an SM slot
// the next layer's decode CTAs could use.
//
// The query and decode kernels use programmatic dependent launch: the
// producers start streaming pages while the query quantizer still runs;
// every thread that reads the packed or raw query or the sink/tail rows, or
// writes the workspace or out, first waits on the preceding grid.
#include <math.h>
#include <stddef.h>

#include <atomic>
#include <mutex>

#include "bd_device.cuh"
#include "bd_query.cuh"

namespace bd {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kConsumers = 4;                    // consumer warps 4..7, one TMEM lane quarter each
constexpr int kFirstConsumer = 4;
constexpr int kThreads = 256;
constexpr int kMaxRec = 9216;                    // one K or V record (NVFP4; MXFP4 is 8704 B)
constexpr int kNK = 4, kNV = 6;                  // K-ring and V-ring slots of kMaxRec bytes
// With the query quantized inside the decode, the rings are filled with the
// first round's four K records and three of its V records (kPreK, kPreV
// pages) before the wait for the preceding grid, the rest after it: later
// pages would only queue, in the memory system, ahead of the preceding grid's
// merge and this grid's query load, and the first round's last V page is
// needed only after its scores.  128K step, one A/B each: all ten slots
// 1238 against 1222 µs for 4 + 4; V pages 0 / 1 / 2 / 3 / 4 with four K
// pages 1228 / 1224 / 1215 / 1212 / 1219; two K pages 1254.
constexpr int kPreK = 4, kPreV = 3;
static_assert(kPreK <= kNK && kPreV <= kNV, "pre-filled pages fit the rings");
constexpr int kCtasPerSm = 2;
// Register split of an FP4 split CTA: launched at kLaunchRegs per thread,
// the control warpgroup gives registers back (setmaxnreg.dec to kCtlRegs)
// and the consumer warpgroup takes them (setmaxnreg.inc to kConsumerRegs).
// The two shares add up exactly to the launch allocation; the host refuses
// to launch if the compiled kernel's register count differs, because an
// increase beyond the launch allocation would wait forever.
constexpr int kLaunchRegs = 128, kCtlRegs = 40, kConsumerRegs = 2 * kLaunchRegs - kCtlRegs;
static_assert(kCtlRegs % 8 == 0 && kConsumerRegs % 8 == 0 && kConsumerRegs <= 256, "setmaxnreg counts");
constexpr int kRingBytes = (kNK + kNV) * kMaxRec;
constexpr int kWavePages = 32;   // one-wave splits up to this many pages ...
constexpr int kBatchPages = 32;  // ... else splits of this many (more if kMaxSplits needs it)
constexpr int kMaxSplits = 64;    // splits + 1 per (sequence, kv head)
constexpr float kSmLog2e = 0.08838834764831845f * 1.4426950408889634f;  // log2(e)/sqrt(128)

// Tensor memory of an FP4 split CTA (256 columns): the score buffer at
// columns 0..127 (one column per token of the page), the query's scale
// factors at 128 (+16 for the second NVFP4 group), and three slots of a
// page's K scale factors at 160 + 32 s (+16).  Every scale-factor address
// starts on a 16-column boundary.
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kSfaCol = 128;
constexpr int kSfbSlots = 3;
static_assert(kSfbSlots < kNK, "a K scale-factor slot's reuse waits on the K ring's empty phases");
__device__ __forceinline__ uint32_t sfb_col(int slot, int j) { return 160u + 32u * slot + 16u * j; }
constexpr int kN = 128;                          // MMA N: the page's tokens
// The query operand: 28 core-matrix groups of 8 rows x 64 B, all zero but
// groups 12 (rows 0..3: term 1 of heads 0..3) and 13 (rows 0..3: term 2).
// For lane quarter w the descriptor starts 4 w groups before group 12, so
// its rows 32 w .. 32 w + 15 are the query and all other rows zero.
constexpr int kQiGroups = 28, kQiFirst = 12;

struct alignas(16) Ctl {
    unsigned long long fullK[kNK], emptyK[kNK];   // K ring (empty: the page's MMAs completed)
    unsigned long long fullV[kNV], emptyV[kNV];   // V ring (empty: the page's consumer warp)
    unsigned long long accFull;                   // a round's scores are in the buffer
    unsigned long long accEmpty;                  // all four consumer warps have read the round
    unsigned long long mmaDone;                   // every MMA the CTA issued has completed
    unsigned long long mergeBar;                  // the merging split's staged partials arrived
    float qred[kThreads / 32];                    // fused query: per-warp amax
    float wm[kConsumers + 1][4];   // per-warp running max per head (log2 units); last: BF16 tokens
    float wl[kConsumers + 1][4];   // per-warp softmax denominator per head
    int abort_flag;
    int last_split;                // this split completed its group's arrival count
    int nlive;                     // split 0 and the splits with pages of this (sequence, kv head)
    int tagK[kNK], tagV[kNV];      // page index each slot's latest fill holds (-1: none)
    int okK[kNK];                  // the K slot's latest fill came from a pool page (published with its tag)
    uint32_t tmem;                 // TMEM base address
};
constexpr int kCtlBytes = (int)((sizeof(Ctl) + 127) / 128 * 128);
constexpr int kTabOff = kRingBytes + kCtlBytes;      // probability-quantizer tables (1 KB)
constexpr int kQiOff = kTabOff + 1024;               // query operand image (28 x 512 B)
constexpr int kSfaOff = kQiOff + kQiGroups * 512;    // query scale-factor groups (2 x 512 B)
constexpr int kQpOff = kSfaOff + 1024;               // fused query: the token's packed query record
constexpr int kFusedMaxHq = 32;                      // fused query quantization up to this many query heads
constexpr int kFusedQpBytes = 4864;                  // the packed record of kFusedMaxHq heads
static_assert(kFusedQpBytes == (kFusedMaxHq * (2 * 64 + 2 * 8 + 4) + 16 + 255) / 256 * 256, "packed query bytes");
constexpr int kSmemBytes = kQpOff + kFusedQpBytes;
static_assert(kCtasPerSm * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");
static_assert(kRingBytes % 128 == 0 && kTabOff % 128 == 0 && kQiOff % 128 == 0 && kSfaOff % 128 == 0 &&
                  kQpOff % 128 == 0 && kMaxRec % 128 == 0,
              "ring slots, tables and operand areas start on 128-byte boundaries");
// Merge area in the (drained) ring: the O of each consumer warp and of the
// BF16 tokens, [kConsumers + 1][4 heads][128] floats; the BF16 staging follows.
constexpr int kStateBytes = (kConsumers + 1) * 4 * 128 * 4;
static_assert(kStateBytes + 143 * 272 + (4 * 128 + 4 * 144) * 4 <= kRingBytes,
              "states and sink/tail staging must fit the ring");

__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint32_t lds16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }

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

// ------------------------------------------------------ BF16 sink + tail --

// Shared-memory row pitch of a staged bf16 head vector: 256 B plus 16 B so
// that eight consecutive rows read with 16-byte loads hit distinct banks.
constexpr int kRowPitch = 272;
constexpr int kMaxBf16Tok = kSink + kPage - 1;   // 143

// Attention of the 4 query heads of kv head h over the BF16 sink and tail
// tokens of sequence b, left as state slot kConsumers of the CTA merge: O in
// the merge area, the maximum and denominator in ctl (maximum -inf: no
// tokens).  Runs on the whole CTA once the ring is no longer in use.
__device__ void tag_counter(const DecodeArgs& a, int b, int h);   // below, with the split merge
__device__ void bf16_segment(const DecodeArgs& a, int b, int h, int L, uint8_t* smem, Ctl* ctl) {
    const int ns = min(L, kSink);
    const int rest = max(0, L - kSink);
    const int npages = rest / kPage;
    const int nt = rest - npages * kPage;
    const int T = ns + nt;
    const int tid = threadIdx.x;
    // the sink/tail rows and q may be produced by the preceding grid
    griddep_wait();
    if (tid == 0) tag_counter(a, b, h);   // thread 0 counts this split in
    if (T <= 0) {
        if (tid < 4) {
            ctl->wm[kConsumers][tid] = -INFINITY;
            ctl->wl[kConsumers][tid] = 0.0f;
        }
        return;
    }
    float* so = reinterpret_cast<float*>(smem) + kConsumers * 4 * kD;   // this state's O
    uint8_t* rows = smem + kStateBytes;                            // [T][272 B] bf16 keys, later values
    float* qf = reinterpret_cast<float*>(rows + kMaxBf16Tok * kRowPitch);   // [4][128]
    float* sp = qf + 4 * kD;                                       // [4][144] scores, then P
    // stage the rows of this kv head (keys now, values after the scores) with
    // asynchronous 16-byte copies (no thread waits for one load before
    // issuing the next)
    auto stage = [&](const uint16_t* sink, const uint16_t* tail) {
        for (int i = tid; i < T * 16; i += blockDim.x) {
            const int tau = i >> 4, c = i & 15;
            const size_t row = tau < ns ? (((size_t)b * kSink + tau) * a.hkv + h) * kD
                                        : (((size_t)b * kPage + (tau - ns)) * a.hkv + h) * kD;
            cp_async16(smem_u32(rows + tau * kRowPitch + 16 * c), (tau < ns ? sink : tail) + row + 8 * c);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    stage(a.sink_k, a.tail_k);
    const uint8_t* ks = rows;
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
    stage(a.sink_v, a.tail_v);   // the keys are no longer read: the values take their place
    const uint8_t* vs = rows;
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
    asm volatile("cp.async.wait_all;" ::: "memory");
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

// ------------------------------------------- FP4 page split: the producers --

// Producer lane: copy page k's K record (isK) or V record into its ring slot
// k % ring size, whose previous fill has been released.
template <int FMT>
__device__ __forceinline__ void fill_slot(const DecodeArgs& a, int h, const int32_t* bt, uint8_t* smem, Ctl* ctl,
                                          bool isK, int k, uint64_t policy) {
    constexpr int RB = (FMT == BD_FORMAT_NVFP4) ? 9216 : 8704;
    const int s = k % (isK ? kNK : kNV);
    const uint32_t full = smem_u32(isK ? &ctl->fullK[s] : &ctl->fullV[s]);
    uint8_t* slot = smem + (isK ? s : kNK + s) * kMaxRec;
    const int64_t phys = bt[k];
    const bool ok = page_ok(phys, a.pool_pages);
    if (isK) ctl->okK[s] = ok ? 1 : 0;   // read by the MMA lane once it has seen the tag
    // tag the fill before it is armed: consumers accept a completed phase
    // only together with their own page index
    st_release_shared(isK ? &ctl->tagK[s] : &ctl->tagV[s], k);
    if (ok) {
        const uint8_t* rec = a.pool + ((phys * a.hkv + h) * 2 + (isK ? 0 : 1)) * (int64_t)RB;
        mbar_arrive_expect_tx(full, RB);
        bulk_g2s_hint(smem_u32(slot), rec, RB, full, policy);
    } else {
        // an entry outside the pool: complete the phase without data
        if (isK) record_error(a.err, BD_ERR_INVALID_ARG);
        mbar_arrive(full);
    }
}

// ------------------------------------------------ FP4 page split: the MMA --

// Lane 0 of warp 2: the query's scale factors into TMEM, then per round of
// four pages (page 4 r + w into lane quarter w) each page's K scale factors
// and its two K = 64 MMAs, S^T = Q K^T with the query operand offset so that
// only quarter w's rows are nonzero.
template <int FMT>
__device__ void mma_rounds(const DecodeArgs& a, int n, const int32_t* bt, uint8_t* smem, Ctl* ctl) {
    constexpr int kGroups = (FMT == BD_FORMAT_NVFP4) ? 2 : 1;
    constexpr uint32_t LBO = 128, SBO = 512;
    const uint32_t tm = ctl->tmem;
    tc_fence_after();
    for (int j = 0; j < kGroups; ++j) tmem_cp_sf(tm + kSfaCol + 16 * j, smem_u32(smem + kSfaOff + 512 * j));
    const uint32_t qimg = smem_u32(smem + kQiOff + kQiFirst * 512);
    const int rounds = (n + 3) / 4;
    bool aborted = false;
    for (int r = 0; r < rounds && !aborted; ++r) {
        // the consumers have read the previous round's scores
        if (r > 0 && !mbar_wait_bounded(smem_u32(&ctl->accEmpty), (r - 1) & 1, kWaitLimitNs, &ctl->abort_flag)) {
            aborted = true;
            break;
        }
        bool first = true;
        for (int w = 0; w < 4; ++w) {
            const int k = 4 * r + w;
            if (k >= n) break;
            const int s = k % kNK, slot = k % kSfbSlots;
            if (!wait_stage_page(smem_u32(&ctl->fullK[s]), (k / kNK) & 1, &ctl->tagK[s], k, &ctl->abort_flag)) {
                aborted = true;
                break;
            }
            // the scale-factor slot's previous MMAs (page k - kSfbSlots) have completed: the empty
            // barrier of that page's K slot says so (its next phase needs the MMAs of page
            // k - kSfbSlots + kNK > k, not issued yet, so the parity cannot alias)
            if (k >= kSfbSlots) {
                const int kp = k - kSfbSlots;
                if (!mbar_wait_bounded(smem_u32(&ctl->emptyK[kp % kNK]), (kp / kNK) & 1, kWaitLimitNs,
                                       &ctl->abort_flag)) {
                    aborted = true;
                    break;
                }
            }
            tc_fence_after();
            if (ctl->okK[s]) {   // published by the producer with the tag wait_stage_page saw
                const uint32_t ks = smem_u32(smem + s * kMaxRec);
                for (int j = 0; j < kGroups; ++j) tmem_cp_sf(tm + sfb_col(slot, j), ks + kCodeBytes + 512 * j);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    // dims 64 j .. 64 j + 63: core-matrix columns 2 j, 2 j + 1
                    const uint64_t ad = smem_desc(qimg - 4 * w * SBO + 2 * j * LBO, LBO, SBO);
                    const uint64_t bdsc = smem_desc(ks + 2 * j * LBO, LBO, SBO);
                    const uint32_t acc = (first && j == 0) ? 0u : 1u;
                    if (FMT == BD_FORMAT_NVFP4) {
                        mma_nvf4(tm, ad, bdsc, mma_idesc_e2m1(kN, false, 0), tm + kSfaCol + 16 * j,
                                 tm + sfb_col(slot, j), acc);
                    } else {
                        // one scale-factor group holds all four 32-dim blocks:
                        // MMA j reads bytes 2 j, 2 j + 1 of each word
                        mma_mxf4(tm, ad, bdsc, mma_idesc_e2m1(kN, true, 2 * j), tm + kSfaCol, tm + sfb_col(slot, 0),
                                 acc);
                    }
                }
                first = false;
                tc_commit(smem_u32(&ctl->emptyK[s]));   // frees the K slot and the scale-factor slot
            } else {
                // an entry outside the pool: no data arrived, nothing to multiply
                mbar_arrive(smem_u32(&ctl->emptyK[s]));
            }
        }
        if (aborted) break;
        tc_commit(smem_u32(&ctl->accFull));
    }
    if (aborted) {
        if (!ctl->abort_flag) record_error(a.err, BD_ERR_TIMEOUT);
        ctl->abort_flag = 1;
    }
    // every MMA issued has finished before the CTA reuses its shared memory
    // or frees the tensor memory
    tc_commit(smem_u32(&ctl->mmaDone));
    (void)mbar_wait_bounded(smem_u32(&ctl->mmaDone), 0, kWaitLimitNs, nullptr);
}

// Warp 2 of an FP4 split CTA.  The whole warp builds the query operand: the
// zero image with group 12 = term 1 and group 13 = term 2 of query heads
// 4h .. 4h+3 (rows 0..3 of each group, core-matrix order: LBO 128 B along K,
// SBO 512 B between groups), and its scale factors as TMEM scale-factor
// groups (lines 0..3 and 8..11, the same word for all four lane quarters).
// Lane 0 then issues the MMAs.
template <int FMT>
__device__ void issue_qk(const DecodeArgs& a, int b, int h, int n, const int32_t* bt, uint8_t* smem, Ctl* ctl,
                         int lane) {
    const uint8_t* qrec;
    if (a.qp) {
        griddep_wait();   // the packed query may come from the preceding grid
        qrec = a.qp + (size_t)b * a.qstride;
    } else {
        qrec = smem + kQpOff;   // quantized by the whole CTA before the roles split
    }
    const int hq = a.hq;
    uint8_t* Qi = smem + kQiOff;
    uint8_t* Sf = smem + kSfaOff;
    for (int i = lane; i < kQiGroups * 512 / 16; i += 32) reinterpret_cast<uint4*>(Qi)[i] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(Sf)[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(Sf)[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    {
        const int row = lane >> 2, ch = lane & 3;   // (term, head) x 4 chunks of 32 dims
        const int term = row >> 2, hh = row & 3;
        *reinterpret_cast<uint4*>(Qi + (kQiFirst + term) * 512 + ch * 128 + hh * 16) =
            *reinterpret_cast<const uint4*>(qrec + (term * hq + 4 * h + hh) * 64 + 16 * ch);
        if (lane < 8) {
            // lane = (term st, head sh); A row 32 w + line: line sh is term 1,
            // line 8 + sh term 2
            const int st = lane >> 2, sh = lane & 3;
            const int line = (st == 0 ? 0 : 8) + sh;
            if (FMT == BD_FORMAT_NVFP4) {
                const uint2 s = *reinterpret_cast<const uint2*>(qrec + 2 * hq * 64 + (st * hq + 4 * h + sh) * 8);
                *reinterpret_cast<uint4*>(Sf + 16 * line) = make_uint4(s.x, s.x, s.x, s.x);         // blocks 0..3
                *reinterpret_cast<uint4*>(Sf + 512 + 16 * line) = make_uint4(s.y, s.y, s.y, s.y);   // blocks 4..7
            } else {
                const uint32_t s = *reinterpret_cast<const uint32_t*>(qrec + 2 * hq * 64 + (st * hq + 4 * h + sh) * 4);
                *reinterpret_cast<uint4*>(Sf + 16 * line) = make_uint4(s, s, s, s);
            }
        }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mma_rounds<FMT>(a, n, bt, smem, ctl);
}

// ------------------------------------------ FP4 page split: the consumers --

// Warps 4..7 of an FP4 split CTA (w = warp - 4): page 4 r + w of every round,
// read from lane quarter w of the score buffer.  Lane (g, t) holds query head
// g (g < 4; rows 4..7 are zero and their lanes compute nothing that is
// read) for the page's tokens 8 j + 2 t + e (j = 0..15, e = 0, 1).  Running
// state per lane: its head's maximum M and its tokens' share of the
// denominator l; O^T as m16n8 accumulator tiles (dims permuted as in the V
// record: lane (g, t) holds dims 16 g .. 16 g + 15 of heads 2 t, 2 t + 1 when
// t < 2).
template <int FMT, int PM>
__device__ void consume_pages(const DecodeArgs& a, const uint8_t* qrec, int h, int n, const int32_t* bt, uint8_t* smem,
                              Ctl* ctl, int w, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const int hq = a.hq;
    const float* gq = reinterpret_cast<const float*>(qrec + 2 * hq * 64 + 2 * hq * 8);
    // score = a1 * (Q1 . K) + a2 * (Q2 . K) + q.mu, in log2 units (MXFP4:
    // the MMA applied every scale already)
    const float a1 = (FMT == BD_FORMAT_NVFP4) ? kSmLog2e * a.gk * gq[0] : kSmLog2e;
    const float a2 = (FMT == BD_FORMAT_NVFP4) ? kSmLog2e * a.gk * gq[1] : kSmLog2e;
    const float bq = a.centering ? kSmLog2e * gq[4 + 4 * h + (g & 3)] : 0.0f;
    const float gV = (FMT == BD_FORMAT_NVFP4) ? a.gv : 1.0f;
    const float ccf = (float)((PM == BD_P_AMAX2_OR_AMAX6) ? a.p_c : 1);
    const float tau = a.tau;
    // per-byte tables (see decode_kernel): [0,128) 1/sd, [128,256) (sd/c, sd/c) f16x2
    const float* ptab_rcp = reinterpret_cast<const float*>(smem + kTabOff);
    const uint32_t* ptab_sdc = reinterpret_cast<const uint32_t*>(ptab_rcp + 128);
    const uint32_t tm_quarter = ctl->tmem + ((uint32_t)(32 * w) << 16);
    // this lane's O columns are heads 2t, 2t+1 (t < 2): lanes 8t and 8t + 4 hold them
    const int srcA = (8 * t) & 31, srcB = (8 * t + 4) & 31;

    float M = -INFINITY, l = 0.0f;
    float o[8][4];
#pragma unroll
    for (int bm = 0; bm < 8; ++bm) o[bm][0] = o[bm][1] = o[bm][2] = o[bm][3] = 0.0f;
    // MXFP4: o holds O / 2^(ref - 127) for this lane's 32-dim V block: ref is
    // the largest V scale byte of that block seen so far (-1: none yet), so
    // every dequantized V value stays at most 6 in f16
    int ref = -1;

    const int rounds = (n + 3) / 4;
    for (int r = 0; r < rounds; ++r) {
        const int k = 4 * r + w;
        const bool has = k < n;
        const bool ok = has && page_ok(bt[k], a.pool_pages);
        if (!mbar_wait_bounded(smem_u32(&ctl->accFull), r & 1, kWaitLimitNs, &ctl->abort_flag)) {
            if (!ctl->abort_flag) record_error(a.err, BD_ERR_TIMEOUT);
            ctl->abort_flag = 1;
            break;
        }
        uint32_t raw[64];
        if (ok) {
            tc_fence_after();
            tmem_ld_16x256b_x16(tm_quarter, raw);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->accEmpty));
        if (!has) continue;
        const int sv = k % kNV;
        if (!ok) {
            // out-of-range block-table entry: no data, the page is left out;
            // hand its V slot back in ring order
            if (!wait_stage_page(smem_u32(&ctl->fullV[sv]), (k / kNV) & 1, &ctl->tagV[sv], k, &ctl->abort_flag)) {
                if (!ctl->abort_flag) record_error(a.err, BD_ERR_TIMEOUT);
                ctl->abort_flag = 1;
                break;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->emptyV[sv]));
            continue;
        }

        // ---------------- scores of head g, tokens 8 j + 2 t + e, log2 units
        float s[32];
#pragma unroll
        for (int j = 0; j < 16; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                s[2 * j + e] = fmaf(__uint_as_float(raw[4 * j + 2 + e]), a2, fmaf(__uint_as_float(raw[4 * j + e]), a1, bq));

        // ---------------- page maximum: 32 in registers, then the 4 lanes t
        float mp = s[0];
#pragma unroll
        for (int i = 1; i < 32; ++i) mp = fmaxf(mp, s[i]);
        mp = fmaxf(mp, __shfl_xor_sync(kFull, mp, 1));
        mp = fmaxf(mp, __shfl_xor_sync(kFull, mp, 2));

        // ---------------- running state: new maximum, page weight, rescale
        const float mn = fmaxf(M, mp);
        const float alpha = ex2(M - mn), wpage = ex2(mp - mn);
        M = mn;
        float pr[32], lp = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            pr[i] = ex2(s[i] - mp);   // P relative to the page's own maximum
            lp += pr[i];
        }
        l = fmaf(l, alpha, wpage * lp);
        const float aA = __shfl_sync(kFull, alpha, srcA), aB = __shfl_sync(kFull, alpha, srcB);
        if (FMT == BD_FORMAT_NVFP4) {   // MXFP4: below, with the V reference
            if (__any_sync(kFull, (aA != 1.0f) | (aB != 1.0f))) {
#pragma unroll
                for (int bm = 0; bm < 8; ++bm) {
                    o[bm][0] *= aA;
                    o[bm][1] *= aB;
                    o[bm][2] *= aA;
                    o[bm][3] *= aB;
                }
            }
        }

        // ---------------- FP4 probabilities: 16-token block i is j = 2i, 2i+1
        // of the four lanes t; the f16x2 of pair j is the P V B-fragment
        // register of k-tile j / 2 (low: token 8 j + 2 t)
        uint32_t ph[16];
        if (PM == BD_P_NONE) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const __half2 hh = __floats2half2_rn(pr[2 * j], pr[2 * j + 1]);
                ph[j] = *reinterpret_cast<const uint32_t*>(&hh);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float u[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) u[e] = pr[4 * i + e] * ccf;
                float bm = fmaxf(fmaxf(u[0], u[1]), fmaxf(u[2], u[3]));
                bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 1));
                bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 2));
                const bool two = (PM == BD_P_AMAX2_OR_AMAX6) && (bm < tau);
                const uint32_t sb = two ? e4m3(bm * 0.5f) : e4m3_div6(bm);
                const float inv = ptab_rcp[sb];   // 0 for the zero scale: all codes 0
                const uint32_t sdc = ptab_sdc[sb];
                ph[2 * i] = hmul2(e2m1x2_to_f16x2(e2m1x2(__fmul_rn(u[0], inv), __fmul_rn(u[1], inv))), sdc);
                ph[2 * i + 1] = hmul2(e2m1x2_to_f16x2(e2m1x2(__fmul_rn(u[2], inv), __fmul_rn(u[3], inv))), sdc);
            }
        }
        {
            // fold the page weight 2^(m_p - M) into Phat: P V accumulates straight into O
            const uint32_t wh = bcast_lo((uint32_t)__half_as_ushort(__float2half_rn(wpage)));
#pragma unroll
            for (int j = 0; j < 16; ++j) ph[j] = hmul2(ph[j], wh);
        }

        // ---------------- P V over the page's eight 16-token groups
        if (!wait_stage_page(smem_u32(&ctl->fullV[sv]), (k / kNV) & 1, &ctl->tagV[sv], k, &ctl->abort_flag)) {
            if (!ctl->abort_flag) record_error(a.err, BD_ERR_TIMEOUT);
            ctl->abort_flag = 1;
            break;
        }
        const uint8_t* Vs = smem + (kNK + sv) * kMaxRec;
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
            // a larger scale in this page raises the reference: o is scaled
            // down by that exact power of two, together with the softmax
            // rescale (a pass of no-op factors is skipped warp-wide)
            const int nref = max(ref, em);
            const int d = ref - nref;
            const float rs = (ref < 0 || d == 0) ? 1.0f : (d < -126 ? 0.0f : pow2i(d));
            ref = nref;
            if (__any_sync(kFull, (aA != 1.0f) | (aB != 1.0f) | (rs != 1.0f))) {
                const float fA = aA * rs, fB = aB * rs;
#pragma unroll
                for (int bm = 0; bm < 8; ++bm) {
                    o[bm][0] *= fA;
                    o[bm][1] *= fB;
                    o[bm][2] *= fA;
                    o[bm][3] *= fB;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // pair rows t and t + 4 of group i hold tokens 16i + 2t, +1 and
            // 16i + 8 + 2t, +1 (k-slots 2t, 2t+1 and 2t+8, 2t+9); dims
            // 16g .. 16g+15 sit at slot g ^ 2t: each quarter warp's eight
            // 16-byte reads cover all 32 banks
            const uint4 v0 = lds128(Vs + (i * 8 + t) * kD + 16 * (g ^ (2 * t)));
            const uint4 v1 = lds128(Vs + (i * 8 + t + 4) * kD + 16 * (g ^ (2 * t)));
            uint32_t vs0, vs1;
            if (FMT == BD_FORMAT_NVFP4) {
                vs0 = e4m3x2_to_f16x2(lds16(Vs + kCodeBytes + ((i * 8 + t) * 8 + g) * 2));
                vs1 = e4m3x2_to_f16x2(lds16(Vs + kCodeBytes + ((i * 8 + t + 4) * 8 + g) * 2));
            } else {
                const uint32_t e0 = lds16(Vs + kCodeBytes + ((i * 8 + t) * 4 + (g >> 1)) * 2);
                const uint32_t e1 = lds16(Vs + kCodeBytes + ((i * 8 + t + 4) * 4 + (g >> 1)) * 2);
                vs0 = f16x2_pow2((int)(e0 & 0xFF) - ref, (int)(e0 >> 8) - ref);
                vs1 = f16x2_pow2((int)(e1 & 0xFF) - ref, (int)(e1 >> 8) - ref);
            }
            const uint32_t b01 = ph[2 * i], b23 = ph[2 * i + 1];
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
                mma16816(o[2 * j], A, b01, b23);
                A[0] = hmul2(f0[2], vs0);
                A[1] = hmul2(f0[3], vs0);
                A[2] = hmul2(f1[2], vs1);
                A[3] = hmul2(f1[3], vs1);
                mma16816(o[2 * j + 1], A, b01, b23);
            }
        }
        // release the V slot: every lane's shared-memory reads are done
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->emptyV[sv]));
    }

    // ---------------- hand the warp state to the CTA merge
    __syncthreads();   // (A) the ring and every MMA are done with
    float* sO = reinterpret_cast<float*>(smem);   // [consumer warps][4 heads][128]
    // NVFP4: the per-tensor V scale; MXFP4: the lane's reference 2^(ref - 127)
    const float gout = (FMT == BD_FORMAT_NVFP4) ? gV : (ref < 0 ? 0.0f : pow2i(ref - 127));
    if (t < 2) {
#pragma unroll
        for (int bm = 0; bm < 8; ++bm) {
            const int d = 16 * g + 2 * bm;
            sO[(w * 4 + 2 * t) * kD + d] = o[bm][0] * gout;
            sO[(w * 4 + 2 * t + 1) * kD + d] = o[bm][1] * gout;
            sO[(w * 4 + 2 * t) * kD + d + 1] = o[bm][2] * gout;
            sO[(w * 4 + 2 * t + 1) * kD + d + 1] = o[bm][3] * gout;
        }
    }
    l += __shfl_xor_sync(kFull, l, 1);
    l += __shfl_xor_sync(kFull, l, 2);
    if (t == 0 && g < 4) {
        ctl->wm[w][g] = M;
        ctl->wl[w][g] = l;
    }
}

// CTA merge of the states (consumer warps, then the BF16 tokens) into this
// split's partial, by 128 threads tid = 0..127 (others pass tid >= 128); a
// state with maximum -inf holds nothing and is skipped.
__device__ void write_split_partial(const DecodeArgs& a, float* part, const uint8_t* smem, const Ctl* ctl, int tid) {
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

// The arrival counter of a (sequence, kv head) group: a word holding the
// call's 40-bit tag over a 24-bit count.  tag_counter runs once per split, by
// the thread that later counts the split in, at the split's start (after the
// dependent-launch wait, so the preceding call's merge is over): a word with
// another tag (an earlier call's, or workspace bytes never written) is
// re-tagged with count 0 by one compare-and-swap.  The swap fails only if a
// split of this call changed the word first, and every such change leaves
// this call's tag in it (tags do not repeat), so whichever split comes
// first, the word holds the tag before any split of the call counts in.
// The read and the swap are thus off the path from a split's last page to
// the merge, where count_split_in is one atomic add, served by the L2
// without retries.
__device__ void tag_counter(const DecodeArgs& a, int b, int h) {
    unsigned long long* cnt = a.counters + (size_t)b * a.hkv + h;
    const unsigned long long w = *reinterpret_cast<volatile unsigned long long*>(cnt);
    if ((w >> 24) != a.tag) atomicCAS(cnt, w, a.tag << 24);
}
// Count this split in; true if it completed the count (nlive arrivals).
__device__ bool count_split_in(const DecodeArgs& a, int b, int h, int nlive) {
    unsigned long long* cnt = a.counters + (size_t)b * a.hkv + h;
    const unsigned long long old = atomicAdd(cnt, 1ull);
    return (old & 0xFFFFFFull) == (unsigned long long)(nlive - 1);   // nlive arrivals in all
}

// Merge the nlive partials (split 0 and the splits with pages) of query heads
// 4h .. 4h+3 of sequence b into out, by 128 threads tid = 0..127 synchronised
// on named barrier 1.  G heads at a time (4 when their records fit the ring
// area, else 2) are staged into shared memory by bulk asynchronous copies,
// one per head (the TMA unit reads L2, where the other SMs' partials are);
// warp hh finds head hh's maximum M over the
// splits with l > 0 (one integer warp reduction of order-preserving keys), the
// weights w_s = 2^(m_s - M) and the denominator sum w_s l_s; each thread then
// sums w_s O_s over its G output dims in split order.  A split with w_s = 0
// wrote no O (its bytes may hold anything, NaN included): it is skipped.
__device__ void merge_group(const DecodeArgs& a, int b, int h, int nlive, uint8_t* smem, Ctl* ctl, int tid) {
    const int nparts = a.nsplit + 1;   // the workspace's record stride per head
    const int lane = tid & 31, warp = tid >> 5;
    const int G = (4 * nlive * kPartStride * 4 <= kRingBytes - 4 * 4 * (kMaxSplits + 1)) ? 4 : 2;
    float* stage = reinterpret_cast<float*>(smem);   // [G][nlive][kPartStride]
    float* sw = stage + G * nlive * kPartStride;   // [G][kMaxSplits] weights, then [G] denominators
    float* sden = sw + G * kMaxSplits;
    const uint32_t bar = smem_u32(&ctl->mergeBar);
    const uint32_t hbytes = (uint32_t)(nlive * kPartStride * 4);   // one head's live records, a multiple of 16
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    // this thread's earlier shared-memory accesses come before the copy's writes
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    for (int h0 = 0, pass = 0; h0 < 4; h0 += G, ++pass) {
        if (tid == 0) {
            mbar_arrive_expect_tx(bar, (uint32_t)G * hbytes);
            for (int hh = 0; hh < G; ++hh)
                bulk_g2s(smem_u32(stage + hh * nlive * kPartStride),
                         a.parts + (size_t)(b * a.hq + 4 * h + h0 + hh) * nparts * kPartStride, hbytes, bar);
        }
        if (!mbar_wait_bounded(bar, pass & 1, kWaitLimitNs, nullptr)) {
            if (tid == 0) record_error(a.err, BD_ERR_TIMEOUT);
            return;   // every thread gives up at the same wait
        }
        if (warp < G) {
            const float* hp = stage + warp * nlive * kPartStride;
            float m[2], l[2];
            uint32_t key = 0;   // order-preserving key of the largest m with l > 0
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int sidx = lane + 32 * r;
                m[r] = (sidx < nlive) ? hp[sidx * kPartStride] : -INFINITY;
                l[r] = (sidx < nlive) ? hp[sidx * kPartStride + 1] : 0.0f;
                if (l[r] > 0.0f) key = max(key, f32_order_key(m[r]));
            }
            key = __reduce_max_sync(kFull, key);
            const float M = (key == 0) ? -INFINITY : f32_from_order_key(key);
            float den = 0.0f;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int sidx = lane + 32 * r;
                const float w = (l[r] > 0.0f) ? ex2(m[r] - M) : 0.0f;
                if (sidx < nlive) sw[warp * kMaxSplits + sidx] = w;
                den = fmaf(w, l[r], den);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
            if (lane == 0) sden[warp] = den;
        }
        named_bar_sync(1, 128);
        // thread tid: head h0 + tid / (128 / G), G consecutive dims
        const int hh = tid / (128 / G), d0 = (tid % (128 / G)) * G;
        const float* hp = stage + hh * nlive * kPartStride + 4 + d0;
        const float* w = sw + hh * kMaxSplits;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        // a split with weight 0 adds exactly 0 (its stored values are finite:
        // zeros when it saw no token), so the loop has no branch and unrolls
#pragma unroll 4
        for (int sidx = 0; sidx < nlive; ++sidx) {
            const float ws = w[sidx];
            if (G == 4) {
                const float4 v = *reinterpret_cast<const float4*>(hp + sidx * kPartStride);
                acc[0] = fmaf(ws, v.x, acc[0]);
                acc[1] = fmaf(ws, v.y, acc[1]);
                acc[2] = fmaf(ws, v.z, acc[2]);
                acc[3] = fmaf(ws, v.w, acc[3]);
            } else {
                const float2 v = *reinterpret_cast<const float2*>(hp + sidx * kPartStride);
                acc[0] = fmaf(ws, v.x, acc[0]);
                acc[1] = fmaf(ws, v.y, acc[1]);
            }
        }
        const float den = sden[hh];
        const float inv = (den > 0.0f) ? 1.0f / den : 0.0f;
        float* o = a.out + ((size_t)b * a.hq + 4 * h + h0 + hh) * kD + d0;
        if (G == 4) {
            *reinterpret_cast<float4*>(o) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
        } else {
            *reinterpret_cast<float2*>(o) = make_float2(acc[0] * inv, acc[1] * inv);
        }
        // the staging area is rewritten by the next pass's copy
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
    }
}

// End of a split, by 128 threads tid = 0..127 (named barrier 1) once each has
// written its share of the split's partial: count the split in and, if it
// was the last of its group, merge the group.
__device__ void finish_split(const DecodeArgs& a, int b, int h, uint8_t* smem, Ctl* ctl, int tid) {
    __threadfence();   // this thread's partial writes are visible device-wide before the count
    // split 0 and the splits with pages (set by thread 0 at the kernel's start)
    const int nlive = ctl->nlive;
    named_bar_sync(1, 128);
    if (tid == 0) ctl->last_split = count_split_in(a, b, h, nlive) ? 1 : 0;
    named_bar_sync(1, 128);
    if (!*reinterpret_cast<volatile int*>(&ctl->last_split)) return;
    __threadfence();   // the other splits' partials, counted in before this one
    merge_group(a, b, h, nlive, smem, ctl, tid);
}

template <int FMT, int PM>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_kernel(const DecodeArgs a) {   // kLaunchRegs
    extern __shared__ __align__(1024) uint8_t smem[];
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

    // a split past its sequence's pages does nothing: it is neither written
    // nor counted, and the merge reads split 0 and the nlive - 1 splits with
    // pages (always the first ones)
    if (p0 >= p1 && !bf16) return;
    if (threadIdx.x == 0) ctl->nlive = 1 + (npages + a.pages_per_split - 1) / a.pages_per_split;
    if (bf16) {
        // no FP4 pages: the consumer states are empty and nothing aborted
        if (threadIdx.x < kConsumers * 4) {
            ctl->wm[threadIdx.x >> 2][threadIdx.x & 3] = -INFINITY;
            ctl->wl[threadIdx.x >> 2][threadIdx.x & 3] = 0.0f;
        }
        if (threadIdx.x == 0) ctl->abort_flag = 0;
        __syncthreads();
        bf16_segment(a, b, h, L, smem, ctl);   // the same for the whole CTA
        __syncthreads();
        write_split_partial(a, part, smem, ctl, threadIdx.x);
        if (threadIdx.x < 128) finish_split(a, b, h, smem, ctl, threadIdx.x);
        return;
    }

    const int n = p1 - p0;
    const int32_t* bt = a.block_table + (size_t)b * a.max_blocks + p0;
    if (warp == 3) tmem_alloc(smem_u32(&ctl->tmem), kTmemCols);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kNK; ++s) {
            mbar_init(smem_u32(&ctl->fullK[s]), 1);
            mbar_init(smem_u32(&ctl->emptyK[s]), 1);
            ctl->tagK[s] = -1;
        }
        for (int s = 0; s < kNV; ++s) {
            mbar_init(smem_u32(&ctl->fullV[s]), 1);
            mbar_init(smem_u32(&ctl->emptyV[s]), 1);   // one consumer warp per page
            ctl->tagV[s] = -1;
        }
        mbar_init(smem_u32(&ctl->accFull), 1);
        mbar_init(smem_u32(&ctl->accEmpty), kConsumers);
        mbar_init(smem_u32(&ctl->mmaDone), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (threadIdx.x >= 128) {
        // exact per-byte tables for the E4M3 scale byte bb: the correctly
        // rounded 1/sd and the f16x2 pair (sd/c, sd/c) for the probability
        // quantizer (exact: c is a power of two)
        float* tab = reinterpret_cast<float*>(smem + kTabOff);
        const uint32_t bb = threadIdx.x - 128;
        const float sd = e4m3_value(bb);
        const float cc = (float)((PM == BD_P_AMAX2_OR_AMAX6) ? a.p_c : 1);
        tab[bb] = (bb == 0) ? 0.0f : __frcp_rn(sd);
        const uint32_t sdh = e4m3x2_to_f16x2(bb);
        const uint32_t icc = bcast_lo((uint32_t)__half_as_ushort(__float2half_rn(1.0f / cc)));
        reinterpret_cast<uint32_t*>(tab)[128 + bb] = hmul2(bcast_lo(sdh), icc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!a.qp) {
        // Fused query: the rings are empty, so the producers fill the first
        // round now (the pages do not depend on the preceding grid); then the whole CTA
        // quantizes this token's query into shared memory -- the bytes
        // bd_quantize_query writes -- one (head, 16-dim chunk) item a thread.
        if (warp < 2 && lane == 0) {
            const bool isK = (warp == 0);
            const uint64_t policy = l2_evict_first_policy();
            for (int k = 0; k < min(n, isK ? kPreK : kPreV); ++k) fill_slot<FMT>(a, h, bt, smem, ctl, isK, k, policy);
        }
        // the warp whose items are this kv head's query heads reads their key
        // mean now: it is in device memory before the kernel starts
        // (bd_set_key_shift returns once it has landed), and a read after the
        // wait would queue behind the ring fill
        qquant::MuPre mu_pre{};
        mu_pre.ok = warp == h && a.centering && a.mu;
        if (mu_pre.ok) {
            const float4* m4 = reinterpret_cast<const float4*>(a.mu + (size_t)h * kD + 16 * (lane & 7));
#pragma unroll
            for (int i = 0; i < 4; ++i) mu_pre.v[i] = m4[i];
        }
        __syncwarp();
        griddep_wait();   // q may come from the preceding grid
        QueryArgs qa;
        qa.q = a.q;
        qa.mu = a.mu;
        qa.qp = nullptr;
        qa.B = a.B;
        qa.hq = a.hq;
        qa.format = FMT;
        qa.rotation = a.rotation;
        qa.centering = a.centering;
        qa.terms = a.terms;
        qa.stride = a.qstride;
        qa.zero_addend = a.zero_addend;
        // the operand image and the consumers need the second term and q.mu
        // of this kv head's query heads only: thread items 32 h .. 32 h + 31,
        // one whole warp
        qquant::quantize_token<1>(qa, a.q + (size_t)b * a.hq * kD, a.mu, smem + kQpOff, (int)threadIdx.x, kThreads,
                                  ctl->qred, [] { __syncthreads(); }, kGroup * h, kGroup * h + kGroup, mu_pre);
        __syncthreads();   // the record is complete
    }
    // Each warpgroup keeps its own register share to the end: the control
    // warpgroup gives registers back, the consumer warpgroup takes them, and
    // the two branches never merge again (code after a merge would have to
    // fit the smaller share).
    static_assert(kCtlRegs == 40 && kConsumerRegs == 216, "the setmaxnreg immediates below");
    if (warp < kFirstConsumer) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 40;" ::: "memory");
        if (warp < 2) {
            // ----------------------------------------------------- producers --
            // warp 0 streams the pages' K records into the K ring, warp 1
            // their V records into the V ring, each in page order
            const bool isK = (warp == 0);
            const int N = isK ? kNK : kNV;
            unsigned long long* fullb = isK ? ctl->fullK : ctl->fullV;
            unsigned long long* emptyb = isK ? ctl->emptyK : ctl->emptyV;
            int* tag = isK ? ctl->tagK : ctl->tagV;
            if (lane == 0) {
                // each page is read once per call: evict it from L2 first
                const uint64_t policy = l2_evict_first_policy();
                // with the fused query the first round was filled before the roles split
                for (int k = a.qp ? 0 : min(n, isK ? kPreK : kPreV); k < n; ++k) {
                    const int s = k % N;
                    if (k >= N && !mbar_wait_bounded(smem_u32(&emptyb[s]), ((k / N) - 1) & 1, kWaitLimitNs,
                                                     &ctl->abort_flag)) {
                        if (!ctl->abort_flag) record_error(a.err, BD_ERR_TIMEOUT);
                        ctl->abort_flag = 1;
                        break;
                    }
                    fill_slot<FMT>(a, h, bt, smem, ctl, isK, k, policy);
                }
            }
            __syncthreads();   // (A)
            // an aborted run drains the copies it left in flight: a slot's last
            // fill is the only one that can be pending
            if (lane == 0 && ctl->abort_flag) {
                for (int s = 0; s < N; ++s) {
                    const int f = tag[s];
                    if (f >= 0) (void)mbar_wait_bounded(smem_u32(&fullb[s]), (f / N) & 1, kWaitLimitNs, nullptr);
                }
            }
        } else if (warp == 2) {
            issue_qk<FMT>(a, b, h, n, bt, smem, ctl, lane);   // the MMA lane waits for its last MMA
            __syncthreads();   // (A)
        } else {
            __syncthreads();   // (A): the consumers' last TMEM loads and every MMA are done
            tc_fence_after();
            tmem_dealloc(ctl->tmem, kTmemCols);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 216;" ::: "memory");
        const int q = warp - kFirstConsumer;
        griddep_wait();   // the packed query may come from the preceding grid
        if (q == 0 && lane == 0) tag_counter(a, b, h);   // the consumer thread that counts this split in
        const uint8_t* qrec = a.qp ? a.qp + (size_t)b * a.qstride : smem + kQpOff;
        consume_pages<FMT, PM>(a, qrec, h, n, bt, smem, ctl, q, lane);   // contains (A)
        if (q == 0 && lane < 4) {   // no BF16 tokens in an FP4 split
            ctl->wm[kConsumers][lane] = -INFINITY;
            ctl->wl[kConsumers][lane] = 0.0f;
        }
        named_bar_sync(1, kConsumers * 32);   // (B) the four warp states are in shared memory
        write_split_partial(a, part, smem, ctl, threadIdx.x - kFirstConsumer * 32);
        finish_split(a, b, h, smem, ctl, threadIdx.x - kFirstConsumer * 32);
    }
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
    // kCtasPerSm CTAs fit per SM; split 0 of every (sequence, kv head) is the
    // BF16 sink/tail CTA, so a single wave holds units * (splits + 1) CTAs.
    // A few slots stay free: while this call's last splits merge, the next
    // call's CTAs (and a separate query quantizer's, launched early) start in
    // them instead of waiting for a slot -- a CTA that starts late holds up
    // its whole layer.  (Measured: no free slot costs 7% at 128K and 38% at
    // 32K; more than eight only lengthens the splits.)
    const int slots = kCtasPerSm * sms - min(max(B, 1), 8);
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

size_t decode_parts_bytes(int B, int hq, int nsplit) {
    return (size_t)B * hq * (nsplit + 1) * kPartStride * sizeof(float);
}

// The workspace: the split partials, one 8-byte arrival counter per
// (sequence, kv head), then (at a 256-byte boundary) room for the packed
// queries a call without a packed query may need (below).
size_t decode_qp_offset(int B, int hq, int hkv, int nsplit) {
    const size_t end = decode_parts_bytes(B, hq, nsplit) + (size_t)B * hkv * sizeof(unsigned long long);
    return (end + 255) / 256 * 256;
}

size_t decode_ws_bytes(int B, int hq, int hkv, int nsplit) {
    return decode_qp_offset(B, hq, hkv, nsplit) + (size_t)B * qpack_stride(hq);
}

// A decode grid that fits one wave (the free slots kept): without a packed
// query, its CTAs quantize the query themselves; a larger grid would repeat
// that in every wave, so the query kernel quantizes it into the workspace
// first.
bool decode_one_wave(int B, int hkv, int nsplit) {
    return (long long)max(1, B * hkv) * (nsplit + 1) <= (long long)kCtasPerSm * device_sms() - min(max(B, 1), 8);
}

unsigned long long next_decode_tag() {
    // Call n gets tag n * K mod 2^40 (K odd: a bijection on 40-bit numbers,
    // so no two of the first 2^40 calls share a tag, and consecutive tags are
    // far apart); tag 0 would be call 2^40 and is skipped.
    static std::atomic<unsigned long long> calls{0};
    for (;;) {
        const unsigned long long n = calls.fetch_add(1) + 1;
        const unsigned long long t = (n * 0x9E3779B97Full) & ((1ull << 40) - 1);
        if (t != 0) return t;
    }
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
            // the register split inside the kernel assumes this launch allocation
            cudaFuncAttributes fa;
            cudaError_t e = cudaFuncGetAttributes(&fa, kern);
            if (e != cudaSuccess) return e;
            if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess) return e;
            g_dev[dev].smem_attr[f][pm] = true;
        }
    }
    DecodeArgs da = a;
    if (!a.qp && !decode_one_wave(a.B, a.hkv, a.nsplit)) {
        QueryArgs qa;
        qa.q = a.q;
        qa.mu = a.mu;
        qa.qp = reinterpret_cast<uint8_t*>(a.parts) + decode_qp_offset(a.B, a.hq, a.hkv, a.nsplit);
        qa.B = a.B;
        qa.hq = a.hq;
        qa.format = a.format;
        qa.rotation = a.rotation;
        qa.centering = a.centering;
        qa.terms = a.terms;
        qa.stride = a.qstride;
        cudaError_t e = launch_query(qa, s);
        if (e != cudaSuccess) return e;
        da.qp = qa.qp;
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
    return cudaLaunchKernelEx(&cfg, kern, da);
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
