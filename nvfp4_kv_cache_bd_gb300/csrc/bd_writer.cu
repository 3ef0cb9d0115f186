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
// (explicit __f*_rn intrinsics, scalar or two-lane packed, so nothing is
// contracted into an FMA; the FMAs that are written out multiply by +-1 and
// round once like the add or subtract they replace); the E2M1 / E4M3
// encodings come from the sm_100-family cvt instructions.
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


// Encode 8 pairs (elements 2i, 2i+1 in xp[i]) with scale (S, inv) into 8
// code bytes (w0: elements 0-7, w1: 8-15) and fill wp[] with the squared
// reconstruction errors of the same pairs.  A zero block encodes with
// inv = 0 and has its codes cleared afterwards: its x_hat is +-0 * S = +-0,
// so its errors are x^2 as for the decoded zero codes.
template <bool kErr>
__device__ __forceinline__ void enc16x2(const float2* xp, float S, float inv, bool zero, float2 z, uint32_t& w0,
                                        uint32_t& w1, float2* wp) {
    const float2 inv2 = splat2(zero ? 0.0f : inv), S2 = splat2(S);
    w0 = 0;
    w1 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t hv;
        const float2 q = mul2(xp[i], inv2);
        const uint32_t byte = e2m1x2_enc_dec(q.x, q.y, hv);
        if (i < 4) w0 |= byte << (8 * i);
        else w1 |= byte << (8 * (i - 4));
        if (kErr) {
            const float2 e = sub2(xp[i], mulz2(f16x2_to_float2(hv), S2, z));
            wp[i] = mulz2(e, e, z);
        }
    }
    if (zero) {
        w0 = 0;
        w1 = 0;
    }
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

// ------------------------------------------------------------------ K tile --

// bf16 x 8 -> four pairs (elements 2i, 2i+1 in xp[i]).
__device__ __forceinline__ void unpack_bf16x8_2(const uint4& u, float2* xp) {
    xp[0] = make_float2(bf16_lo(u.x), bf16_hi(u.x));
    xp[1] = make_float2(bf16_lo(u.y), bf16_hi(u.y));
    xp[2] = make_float2(bf16_lo(u.z), bf16_hi(u.z));
    xp[3] = make_float2(bf16_lo(u.w), bf16_hi(u.w));
}

// A lane's 16 dims are held as 8 pairs xp[i] = (x[2i], x[2i+1]); every step
// below is the scalar sequence of the transform and the search, two
// elements per packed instruction where both take the same operation.
template <int FMT>
__device__ void write_k_tile(const WriterArgs& a, const uint8_t* tile, int row0, const float* stab, uint8_t* rec,
                             int grp, int lane, int h) {
    const int r = lane >> 3, c = lane & 7;
    const float2 z = splat2(a.zero_addend);
    float2 mu[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        mu[i] = (a.centering && a.mu) ? make_float2(a.mu[h * kD + 16 * c + 2 * i], a.mu[h * kD + 16 * c + 2 * i + 1])
                                      : make_float2(0.0f, 0.0f);

#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
        const int tok = 16 * grp + 4 * j + r;
        float2 xp[8];
        unpack_bf16x8_2(lds128(tile + (tok - row0) * kTilePitch + 32 * c), xp);
        unpack_bf16x8_2(lds128(tile + (tok - row0) * kTilePitch + 32 * c + 16), xp + 4);
        if (a.centering) {
#pragma unroll
            for (int i = 0; i < 8; ++i) xp[i] = sub2(xp[i], mu[i]);
        }
        if (a.rotation) {
            // stride 1 inside each pair
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float u = xp[i].x, v = xp[i].y;
                xp[i] = make_float2(__fadd_rn(u, v), __fsub_rn(u, v));
            }
            // strides 2, 4, 8 between pairs
#pragma unroll
            for (int hs = 1; hs < 8; hs <<= 1)
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (!(i & hs)) {
                        const float2 u = xp[i], v = xp[i + hs];
                        xp[i] = add2(u, v);
                        xp[i + hs] = sub2(u, v);
                    }
            // strides 16, 32, 64 across lanes c^1, c^2, c^4
#pragma unroll
            for (int m = 1; m <= 4; m <<= 1) {
                // p - x in the upper lane, x + p in the lower one: fma(x, +-1, p)
                // rounds the exact p +- x once, like the add or subtract
                const float2 sgn = splat2((c & m) ? -1.0f : 1.0f);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 p = make_float2(__shfl_xor_sync(kFull, xp[i].x, m), __shfl_xor_sync(kFull, xp[i].y, m));
                    xp[i] = fma2(xp[i], sgn, p);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) xp[i] = mulz2(xp[i], splat2(kRot), z);
        }

        uint32_t w0, w1, sb;
        float2 wp[8];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(xp[i].x), fabsf(xp[i].y)));
        if (FMT == BD_FORMAT_NVFP4) {
            Scale s6 = nv_scale(amax, 6.0f, a.gk, stab);
            if (a.key_search) {
                uint32_t c0, c1;
                enc16x2<true>(xp, s6.S, s6.inv, s6.zero, z, c0, c1, wp);
                const float e6 = tree16x2(wp);
                Scale s4 = nv_scale(amax, 4.0f, a.gk, stab);
                enc16x2<true>(xp, s4.S, s4.inv, s4.zero, z, w0, w1, wp);
                const float e4 = tree16x2(wp);
                sb = s4.sb;
                if (!(e4 < e6)) { w0 = c0; w1 = c1; sb = s6.sb; }
            } else {
                enc16x2<false>(xp, s6.S, s6.inv, s6.zero, z, w0, w1, wp);
                sb = s6.sb;
            }
        } else {
            // The 32-element block spans lanes c and c^1; every lane runs the
            // same shuffles (a zero block takes its result from the select).
            const float amax32 = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
            int ea, eb;
            mx_candidates(amax32 == 0.0f ? 1.0f : amax32, ea, eb);
            uint32_t c0, c1;
            mx_enc_err16x2(xp, ea, z, c0, c1, wp);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                wp[i] = add2(wp[i], make_float2(__shfl_xor_sync(kFull, wp[i].x, 1), __shfl_xor_sync(kFull, wp[i].y, 1)));
            const float sa = tree16x2(wp);
            mx_enc_err16x2(xp, eb, z, w0, w1, wp);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                wp[i] = add2(wp[i], make_float2(__shfl_xor_sync(kFull, wp[i].x, 1), __shfl_xor_sync(kFull, wp[i].y, 1)));
            const float sbb = tree16x2(wp);
            // the codes of the chosen candidate; a zero block has codes 0
            const int e = (amax32 == 0.0f) ? -127 : ((sbb < sa) ? eb : ea);
            if (!(sbb < sa)) { w0 = c0; w1 = c1; }
            if (amax32 == 0.0f) { w0 = 0; w1 = 0; }
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

// bf16 x 8 of two tokens -> eight (token 0, token 1) pairs of the same dims.
__device__ __forceinline__ void unpack_rows_2(const uint4& u0, const uint4& u1, float2* xv) {
    xv[0] = make_float2(bf16_lo(u0.x), bf16_lo(u1.x));
    xv[1] = make_float2(bf16_hi(u0.x), bf16_hi(u1.x));
    xv[2] = make_float2(bf16_lo(u0.y), bf16_lo(u1.y));
    xv[3] = make_float2(bf16_hi(u0.y), bf16_hi(u1.y));
    xv[4] = make_float2(bf16_lo(u0.z), bf16_lo(u1.z));
    xv[5] = make_float2(bf16_hi(u0.z), bf16_hi(u1.z));
    xv[6] = make_float2(bf16_lo(u0.w), bf16_lo(u1.w));
    xv[7] = make_float2(bf16_hi(u0.w), bf16_hi(u1.w));
}

// Encode 16 dims of two tokens (xv[d] = (token 0, token 1)) into 16 paired
// code bytes, token 0 in the low nibble: inv holds each token's 1/S.
__device__ __forceinline__ void enc_pairs16(const float2* xv, float2 inv, uint32_t* words) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t wd = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float2 v = mul2(xv[4 * q + b], inv);
            wd |= e2m1x2(v.x, v.y) << (8 * b);
        }
        words[q] = wd;
    }
}

// Code-word mask that clears the nibbles of zero blocks (token 0's are the
// low nibbles): their codes are 0, whatever the sign of the encoded zeros.
__device__ __forceinline__ uint32_t zero_mask(bool z0, bool z1) {
    return (z0 ? 0xF0F0F0F0u : 0xFFFFFFFFu) & (z1 ? 0x0F0F0F0Fu : 0xFFFFFFFFu);
}

// One MXFP4 candidate for the 32-dim blocks of two tokens at once, exponent
// e.x for token 0 and e.y for token 1: the 32 paired code bytes and both
// squared-error sums, each summed as w[i] = err(i) + err(16+i), then the
// tree levels w[i] += w[i+8], +4, +2, +1.
__device__ __forceinline__ float2 mx_pair_cand32(const float2* xv, int e0, int e1, float2 z, uint32_t* words) {
    const float2 down = make_float2(pow2i(-e0), pow2i(-e1)), up = make_float2(pow2i(e0), pow2i(e1));
    float2 w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) words[q] = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float2 t[4];   // dims i, 16+i, 8+i, 24+i
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int d = i + (k == 1 ? 16 : k == 2 ? 8 : k == 3 ? 24 : 0);
            uint32_t hv;
            const float2 v = mul2(xv[d], down);
            words[d >> 2] |= e2m1x2_enc_dec(v.x, v.y, hv) << (8 * (d & 3));
            const float2 err = sub2(xv[d], mulz2(f16x2_to_float2(hv), up, z));
            t[k] = mulz2(err, err, z);
        }
        w[i] = add2(add2(t[0], t[1]), add2(t[2], t[3]));
    }
#pragma unroll
    for (int h = 4; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) w[i] = add2(w[i], w[i + h]);
    return w[0];
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
            float2 xv[16];
            unpack_rows_2(lds128(r0 + 32 * blk), lds128(r1 + 32 * blk), xv);
            unpack_rows_2(lds128(r0 + 32 * blk + 16), lds128(r1 + 32 * blk + 16), xv + 8);
            float am0 = 0.0f, am1 = 0.0f;
#pragma unroll
            for (int d = 0; d < 16; ++d) {
                am0 = fmaxf(am0, fabsf(xv[d].x));
                am1 = fmaxf(am1, fabsf(xv[d].y));
            }
            Scale s0 = nv_scale(am0, 6.0f, a.gv, stab);
            Scale s1 = nv_scale(am1, 6.0f, a.gv, stab);
            enc_pairs16(xv, make_float2(s0.zero ? 0.0f : s0.inv, s1.zero ? 0.0f : s1.inv), words + 4 * blk);
            const uint32_t m = zero_mask(s0.zero, s1.zero);
#pragma unroll
            for (int q = 0; q < 4; ++q) words[4 * blk + q] &= m;
            sbs |= (s0.sb | (s1.sb << 8)) << (16 * blk);
        }
        *reinterpret_cast<uint32_t*>(rec + kCodeBytes + ((grp * 8 + p) * 8 + 2 * c) * 2) = sbs;
    } else {
        float2 xv[32];
#pragma unroll
        for (int k = 0; k < 4; ++k) unpack_rows_2(lds128(r0 + 16 * k), lds128(r1 + 16 * k), xv + 8 * k);
        float am0 = 0.0f, am1 = 0.0f;
#pragma unroll
        for (int d = 0; d < 32; ++d) {
            am0 = fmaxf(am0, fabsf(xv[d].x));
            am1 = fmaxf(am1, fabsf(xv[d].y));
        }
        const bool z0 = am0 == 0.0f, z1 = am1 == 0.0f;   // zero blocks: codes 0, scale byte 0
        int ea0, eb0, ea1, eb1;
        mx_candidates(z0 ? 1.0f : am0, ea0, eb0);
        mx_candidates(z1 ? 1.0f : am1, ea1, eb1);
        uint32_t wb[8];
        const float2 z = splat2(a.zero_addend);
        const float2 sa = mx_pair_cand32(xv, ea0, ea1, z, words);
        const float2 sbb = mx_pair_cand32(xv, eb0, eb1, z, wb);
        const bool b0 = sbb.x < sa.x, b1 = sbb.y < sa.y;   // the larger exponent only when strictly better
        const uint32_t mb = (b0 ? 0x0F0F0F0Fu : 0u) | (b1 ? 0xF0F0F0F0u : 0u), mz = zero_mask(z0, z1);
#pragma unroll
        for (int q = 0; q < 8; ++q) words[q] = ((words[q] & ~mb) | (wb[q] & mb)) & mz;
        const uint32_t s0 = z0 ? 0u : (uint32_t)((b0 ? eb0 : ea0) + 127);
        const uint32_t s1 = z1 ? 0u : (uint32_t)((b1 ? eb1 : ea1) + 127);
        *reinterpret_cast<uint16_t*>(rec + kCodeBytes + ((grp * 8 + p) * 4 + c) * 2) = (uint16_t)(s0 | (s1 << 8));
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
