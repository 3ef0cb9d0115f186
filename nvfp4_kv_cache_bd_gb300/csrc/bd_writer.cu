// Page-fill writer: quantizes freshly filled 128-token KV pages into the
// packed NVFP4 / MXFP4 pool records.
//
// Method: BitDecoding-FP4 evaluation config (config.py) RECIPE
// outlier_aware_key_quantization (key smoothing, Hadamard rotation, adaptive
// {4,6} block-scale search), recipe_additional_config (value scale mode
// "amax6"), KV_MODES["bitdecoding-mxfp4"] scale_mode "mxfp4_search";
// freeze-at-fill pages from kv-landlords quant_ab.py (module docstring).
//
// Grid: one CTA of 4 warps per (page, kv head, half page, K or V), the key
// CTAs first in launch order.  The CTA
// first stages its 64 bf16 rows in shared memory with coalesced 16-byte
// asynchronous copies; each warp then owns one 16-token x 128-dim tile and
// reads its lanes' values from there.
//  K warp: lane = (token r = lane/8 of 4, 16-dim chunk c = lane%8).  The
//    Hadamard transform runs strides 1..8 inside a lane and strides 16, 32,
//    64 across lanes c^1, c^2, c^4 by warp shuffles; an NVFP4 block (16 dims)
//    is then entirely in one lane, an MXFP4 block (32 dims) in a lane pair.
//  V warp: lane = (token pair p = lane%8: tokens 16i+2p and 16i+2p+1, 32-dim
//    chunk c = lane/8), so both nibbles of a V code byte are produced in the
//    same lane and the 16-token tile is written with 16-byte stores.
// Every rounding step is the IEEE binary32 operation the oracle performs
// (explicit __f*_rn intrinsics, so nothing is contracted into an FMA; the
// one FMA, in the cross-lane butterflies, multiplies by +-1 and rounds once
// like the add it replaces); the E2M1 / E4M3 encodings come from the
// sm_100-family cvt instructions.
#include "bd_device.cuh"

namespace bd {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
// Staged bf16 rows: 256 B plus 16 B, so that both lane layouts read their
// 16-byte pieces from distinct banks (4 lanes per 4-bank group).
constexpr int kTilePitch = 272;
// A CTA covers half a page (64 tokens, 4 warps of 16): small CTAs spread the
// heavy key tiles evenly over the SMs.
constexpr int kCtaRows = 64;
constexpr int kCtaThreads = 2 * kCtaRows;
constexpr int kTileBytes = kCtaRows * kTilePitch;
constexpr int kSTabBytes = 2 * 128 * 4;   // NVFP4 scale tables after the tile

struct Scale {
    uint32_t sb;
    float S, inv;
    bool zero;
};

// NVFP4 scale of a block: t = m*g, s = amax/t -> E4M3 byte, S = E4M3*g, 1/S.
// stab holds S and RN(1/S) for every byte (scale_tables); s >= 0, so the
// byte is below 128.
__device__ __forceinline__ Scale nv_scale(float amax, float m, float g, const float* stab) {
    Scale r;
    float t = __fmul_rn(m, g);
    float s = __fdiv_rn(amax, t);
    r.sb = e4m3(s);
    r.S = stab[r.sb];
    r.inv = stab[128 + r.sb];
    r.zero = (r.S == 0.0f) || isinf(r.inv);
    return r;
}

// Per-CTA tables for the CTA's per-tensor scale g: S_b = E4M3(b) * g and its
// correctly rounded reciprocal, for the 128 non-negative scale bytes b.
__device__ __forceinline__ void scale_tables(float g, float* stab) {
    if (threadIdx.x < 128) {
        const float S = __fmul_rn(e4m3_value(threadIdx.x), g);
        stab[threadIdx.x] = S;
        stab[128 + threadIdx.x] = __frcp_rn(S);
    }
}

// Two values -> one byte of E2M1 codes (lo in bits 3..0), and that byte
// decoded back to f16x2 (exact), from one conversion register.
__device__ __forceinline__ uint32_t e2m1x2_enc_dec(float lo, float hi, uint32_t& f16x2) {
    uint32_t byte, h;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %3;\n\tcvt.rn.f16x2.e2m1x2 %1, t;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(byte), "=r"(h)
        : "f"(hi), "f"(lo));
    f16x2 = h;
    return byte;
}

// Squared-error tree over 16 terms: w[i] += w[i+8], then +4, +2, +1.
__device__ __forceinline__ float tree16(float* w) {
#pragma unroll
    for (int h = 8; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) w[i] = __fadd_rn(w[i], w[i + h]);
    return w[0];
}

// Encode 16 values with scale (S, inv) into 8 code bytes (w0: elements 0-7,
// w1: 8-15) and fill w[] with squared reconstruction errors.
template <bool kErr>
__device__ __forceinline__ void enc16(const float* x, float S, float inv, bool zero, uint32_t& w0,
                                      uint32_t& w1, float* w) {
    w0 = 0;
    w1 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t byte = 0, hv = 0;
        if (!zero) byte = e2m1x2_enc_dec(__fmul_rn(x[2 * i], inv), __fmul_rn(x[2 * i + 1], inv), hv);
        if (i < 4) w0 |= byte << (8 * i);
        else w1 |= byte << (8 * (i - 4));
        if (kErr) {
            // a zero block decodes to 0 and S is finite, so x_hat = 0 * S = +0
            const float2 val = f16x2_to_float2(hv);
            const float e0 = __fsub_rn(x[2 * i], __fmul_rn(val.x, S));
            const float e1 = __fsub_rn(x[2 * i + 1], __fmul_rn(val.y, S));
            w[2 * i] = __fmul_rn(e0, e0);
            w[2 * i + 1] = __fmul_rn(e1, e1);
        }
    }
}

__device__ __forceinline__ float amax_of(const float* x, int n) {
    float a = 0.0f;
    for (int i = 0; i < n; ++i) a = fmaxf(a, fabsf(x[i]));
    return a;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* x) {
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x);
    x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z);
    x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
    return *reinterpret_cast<const uint4*>(p);
}

// MXFP4 candidates e0 = floor(log2 amax) - 2 and e0 + 1, clamped to [-127,127].
__device__ __forceinline__ void mx_candidates(float amax, int& ea, int& eb) {
    int E = ilog2f(amax);
    ea = min(127, max(-127, E - 2));
    eb = min(127, max(-127, E - 1));
}

// Squared errors of 16 values quantized with exponent e.
__device__ __forceinline__ void mx_err16(const float* x, int e, float* w) {
    float down = pow2i(-e), up = pow2i(e);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t byte = e2m1x2(__fmul_rn(x[2 * i], down), __fmul_rn(x[2 * i + 1], down));
        float2 val = f16x2_to_float2(e2m1x2_to_f16x2(byte));
        float e0 = __fsub_rn(x[2 * i], __fmul_rn(val.x, up));
        float e1 = __fsub_rn(x[2 * i + 1], __fmul_rn(val.y, up));
        w[2 * i] = __fmul_rn(e0, e0);
        w[2 * i + 1] = __fmul_rn(e1, e1);
    }
}

// ------------------------------------------------------------------ K tile --

template <int FMT>
__device__ void write_k_tile(const WriterArgs& a, const uint8_t* tile, int row0, const float* stab, uint8_t* rec,
                             int grp, int lane, int h) {
    const int r = lane >> 3, c = lane & 7;
    float mu[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) mu[i] = (a.centering && a.mu) ? a.mu[h * kD + 16 * c + i] : 0.0f;

#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
        const int tok = 16 * grp + 4 * j + r;
        float x[16];
        unpack_bf16x8(lds128(tile + (tok - row0) * kTilePitch + 32 * c), x);
        unpack_bf16x8(lds128(tile + (tok - row0) * kTilePitch + 32 * c + 16), x + 8);
        if (a.centering) {
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = __fsub_rn(x[i], mu[i]);
        }
        if (a.rotation) {
            // strides 1, 2, 4, 8 inside the lane
#pragma unroll
            for (int hs = 1; hs < 16; hs <<= 1)
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (!(i & hs)) {
                        float u = x[i], v = x[i + hs];
                        x[i] = __fadd_rn(u, v);
                        x[i + hs] = __fsub_rn(u, v);
                    }
            // strides 16, 32, 64 across lanes c^1, c^2, c^4
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

        uint32_t w0, w1, sb;
        float w[16];
        const float amax = amax_of(x, 16);
        if (FMT == BD_FORMAT_NVFP4) {
            Scale s6 = nv_scale(amax, 6.0f, a.gk, stab);
            if (a.key_search) {
                uint32_t c0, c1;
                enc16<true>(x, s6.S, s6.inv, s6.zero, c0, c1, w);
                const float e6 = tree16(w);
                Scale s4 = nv_scale(amax, 4.0f, a.gk, stab);
                enc16<true>(x, s4.S, s4.inv, s4.zero, w0, w1, w);
                const float e4 = tree16(w);
                sb = s4.sb;
                if (!(e4 < e6)) { w0 = c0; w1 = c1; sb = s6.sb; }
            } else {
                enc16<false>(x, s6.S, s6.inv, s6.zero, w0, w1, w);
                sb = s6.sb;
            }
        } else {
            // The 32-element block spans lanes c and c^1; every lane runs the
            // same shuffles (a zero block takes its result from the select).
            const float amax32 = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
            int ea, eb;
            mx_candidates(amax32 == 0.0f ? 1.0f : amax32, ea, eb);
            mx_err16(x, ea, w);
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __fadd_rn(w[i], __shfl_xor_sync(kFull, w[i], 1));
            const float sa = tree16(w);
            mx_err16(x, eb, w);
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __fadd_rn(w[i], __shfl_xor_sync(kFull, w[i], 1));
            const float sbb = tree16(w);
            const int e = (amax32 == 0.0f) ? -127 : ((sbb < sa) ? eb : ea);
            const float down = pow2i(-e);
            enc16<false>(x, 0.0f, down, amax32 == 0.0f, w0, w1, w);
            sb = (amax32 == 0.0f) ? 0u : (uint32_t)(e + 127);
        }
        // codes in groups of 8 tokens x 32 dims (128 B each); scale byte of
        // block b at (b/4)*512 + (tok%32)*16 + (tok/32)*4 + b%4
        *reinterpret_cast<uint2*>(rec + (tok >> 3) * 512 + (c >> 1) * 128 + (tok & 7) * 16 + 8 * (c & 1)) =
            make_uint2(w0, w1);
        const int sline = kCodeBytes + (tok & 31) * 16 + (tok >> 5) * 4;
        if (FMT == BD_FORMAT_NVFP4) rec[sline + (c >> 2) * 512 + (c & 3)] = (uint8_t)sb;
        else if (!(c & 1)) rec[sline + (c >> 1)] = (uint8_t)sb;
    }
}

// ------------------------------------------------------------------ V tile --

// Encode the same 16 dims of two tokens into 16 paired code bytes.
__device__ __forceinline__ void enc_pair16(const float* x0, const float* x1, float inv0, bool z0, float inv1,
                                           bool z1, uint32_t* words) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t wd = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int d = 4 * q + b;
            const float lo = z0 ? 0.0f : __fmul_rn(x0[d], inv0);
            const float hi = z1 ? 0.0f : __fmul_rn(x1[d], inv1);
            wd |= e2m1x2(lo, hi) << (8 * b);
        }
        words[q] = wd;
    }
}

__device__ __forceinline__ int mx_search32(const float* x) {
    const float amax = amax_of(x, 32);
    if (amax == 0.0f) return -128;   // marker: zero block
    int ea, eb;
    mx_candidates(amax, ea, eb);
    float w[16], w2[16];
    mx_err16(x, ea, w);
    mx_err16(x + 16, ea, w2);
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = __fadd_rn(w[i], w2[i]);
    const float sa = tree16(w);
    mx_err16(x, eb, w);
    mx_err16(x + 16, eb, w2);
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = __fadd_rn(w[i], w2[i]);
    const float sbb = tree16(w);
    return (sbb < sa) ? eb : ea;
}

template <int FMT>
__device__ void write_v_tile(const WriterArgs& a, const uint8_t* tile, int row0, const float* stab, uint8_t* rec,
                             int grp, int lane) {
    const int p = lane & 7, c = lane >> 3;
    const int t0 = 16 * grp + 2 * p, t1 = t0 + 1;
    const uint8_t* r0 = tile + (t0 - row0) * kTilePitch + 64 * c;   // dims 32c .. 32c+31 of both tokens
    const uint8_t* r1 = tile + (t1 - row0) * kTilePitch + 64 * c;
    // dims 32c .. 32c+31 are 16-byte slots 2c, 2c+1, stored at slots
    // 2c XOR 2(p mod 4) and the one after it
    uint8_t* codes = rec + (grp * 8 + p) * kD + 32 * (c ^ (p & 3));
    uint32_t words[8];
    if (FMT == BD_FORMAT_NVFP4) {
        // one 16-dim block of both tokens at a time
        uint32_t sbs = 0;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
            float x0[16], x1[16];
            unpack_bf16x8(lds128(r0 + 32 * blk), x0);
            unpack_bf16x8(lds128(r0 + 32 * blk + 16), x0 + 8);
            unpack_bf16x8(lds128(r1 + 32 * blk), x1);
            unpack_bf16x8(lds128(r1 + 32 * blk + 16), x1 + 8);
            Scale s0 = nv_scale(amax_of(x0, 16), 6.0f, a.gv, stab);
            Scale s1 = nv_scale(amax_of(x1, 16), 6.0f, a.gv, stab);
            enc_pair16(x0, x1, s0.inv, s0.zero, s1.inv, s1.zero, words + 4 * blk);
            sbs |= (s0.sb | (s1.sb << 8)) << (16 * blk);
        }
        *reinterpret_cast<uint32_t*>(rec + kCodeBytes + ((grp * 8 + p) * 8 + 2 * c) * 2) = sbs;
    } else {
        float x0[32], x1[32];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            unpack_bf16x8(lds128(r0 + 16 * k), x0 + 8 * k);
            unpack_bf16x8(lds128(r1 + 16 * k), x1 + 8 * k);
        }
        const int e0 = mx_search32(x0), e1 = mx_search32(x1);
        const bool z0 = e0 == -128, z1 = e1 == -128;
        const float d0 = z0 ? 0.0f : pow2i(-e0), d1 = z1 ? 0.0f : pow2i(-e1);
        enc_pair16(x0, x1, d0, z0, d1, z1, words);
        enc_pair16(x0 + 16, x1 + 16, d0, z0, d1, z1, words + 4);
        const uint32_t b0 = z0 ? 0u : (uint32_t)(e0 + 127), b1 = z1 ? 0u : (uint32_t)(e1 + 127);
        *reinterpret_cast<uint16_t*>(rec + kCodeBytes + ((grp * 8 + p) * 4 + c) * 2) = (uint16_t)(b0 | (b1 << 8));
    }
    *reinterpret_cast<uint4*>(codes) = make_uint4(words[0], words[1], words[2], words[3]);
    *reinterpret_cast<uint4*>(codes + 16) = make_uint4(words[4], words[5], words[6], words[7]);
}

// NVFP4 fits eight CTAs per SM (64 registers); MXFP4 value blocks keep a
// whole 32-element block of two tokens in registers.
template <int FMT>
__global__ void __launch_bounds__(kCtaThreads, FMT == BD_FORMAT_NVFP4 ? 8 : 4) writer_kernel(const WriterArgs a) {
    extern __shared__ __align__(16) uint8_t tile[];   // [kCtaRows tokens][kTilePitch]: this head's bf16 rows
    // grid (pages x heads, half page, K or V): every K CTA comes before every
    // V CTA in launch order, so the heavy key tiles all start in the first
    // wave and the light value tiles fill the slots they leave
    const int pg = blockIdx.x / a.hkv, h = blockIdx.x % a.hkv;
    const int kv = blockIdx.z;
    const int half = blockIdx.y;
    const int row0 = kCtaRows * half;                  // first token of this CTA's half page
    const int grp = (row0 >> 4) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const size_t tok_stride = (size_t)a.hkv * kD;
    int64_t page;
    const uint16_t* newrow = nullptr;   // append mode: the new token's row, staged as the page's last row
    const bool reporter = threadIdx.x == 0 && kv == 0 && half == 0;   // one report per page
    if (a.seq_lens) {
        // append the token at position L (pg is the sequence) ...
        const int L = a.seq_lens[pg];
        if (L < 0) {
            if (reporter && h == 0) record_error(a.err, BD_ERR_INVALID_ARG);
            return;
        }
        const uint16_t* nrow = (kv == 0 ? a.k_new : a.v_new) + ((size_t)pg * a.hkv + h) * kD;
        if (L < kSink) {
            uint16_t* dst = (kv == 0 ? a.sink_k : a.sink_v) + (((size_t)pg * kSink + L) * a.hkv + h) * kD;
            if (half == 0 && threadIdx.x < 16)
                reinterpret_cast<uint4*>(dst)[threadIdx.x] = reinterpret_cast<const uint4*>(nrow)[threadIdx.x];
            return;
        }
        const int r = (L - kSink) % kPage, p = (L - kSink) / kPage;
        if (r / kCtaRows == half && threadIdx.x < 16) {
            uint16_t* dst = (kv == 0 ? a.tail_k : a.tail_v) + (((size_t)pg * kPage + r) * a.hkv + h) * kD;
            reinterpret_cast<uint4*>(dst)[threadIdx.x] = reinterpret_cast<const uint4*>(nrow)[threadIdx.x];
        }
        // ... and pack the tail page it completes
        if (r != kPage - 1) return;
        if (p >= a.max_blocks) {
            if (reporter) record_error(a.err, BD_ERR_INVALID_ARG);
            return;
        }
        page = a.block_table[(size_t)pg * a.max_blocks + p];
        newrow = nrow;
    } else {
        page = a.dst_pages[pg];
    }
    if (!page_ok(page, a.pool_pages)) {   // never write outside the pool
        if (reporter) record_error(a.err, BD_ERR_INVALID_ARG);
        return;
    }
    uint8_t* rec = a.pool + ((page * a.hkv + h) * 2 + kv) * (int64_t)record_bytes(a.format);
    const uint16_t* src = (kv == 0 ? a.k : a.v) + (((size_t)pg * kPage + row0) * a.hkv + h) * kD;
    // stage the CTA's rows (256 B each) with coalesced 16-byte copies
    for (int q = threadIdx.x; q < kCtaRows * 16; q += blockDim.x) {
        const int row = q >> 4, ch = q & 15;
        const uint16_t* from = (newrow && row0 + row == kPage - 1) ? newrow + 8 * ch
                                                                     : src + (size_t)row * tok_stride + 8 * ch;
        cp_async16(smem_u32(tile + row * kTilePitch + 16 * ch), from);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    float* stab = reinterpret_cast<float*>(tile + kTileBytes);
    if (FMT == BD_FORMAT_NVFP4) scale_tables(kv == 0 ? a.gk : a.gv, stab);   // while the copies fly
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (kv == 0) write_k_tile<FMT>(a, tile, row0, stab, rec, grp, lane, h);
    else write_v_tile<FMT>(a, tile, row0, stab, rec, grp, lane);
}

}  // namespace

cudaError_t launch_writer(const WriterArgs& a, cudaStream_t s) {
    if (a.n == 0) return cudaSuccess;
    dim3 grid((unsigned)(a.n * a.hkv), kPage / kCtaRows, 2);
    if (a.format == BD_FORMAT_NVFP4)
        writer_kernel<BD_FORMAT_NVFP4><<<grid, kCtaThreads, kTileBytes + kSTabBytes, s>>>(a);
    else
        writer_kernel<BD_FORMAT_MXFP4><<<grid, kCtaThreads, kTileBytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace bd
