// Device helpers for the sm_103a kernels: FP4/FP8 conversions through the
// hardware cvt instructions, exact IEEE arithmetic without contraction,
// mbarrier + bulk-copy (TMA) primitives with bounded waits, and the
// m16n8k16 f16 tensor-core MMA.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "bd_internal.h"

namespace bd {

constexpr float kRot = 0.08838834764831845f;   // binary32(1/sqrt(128)) = 0x3DB504F3
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- formats --

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two binary32 values -> one byte of two E2M1 codes (lo in bits 3..0, hi in
// bits 7..4); round to nearest even, saturating at +-6.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// One byte of two E2M1 codes -> f16x2 (low nibble -> low half).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    uint16_t b = (uint16_t)byte;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "h"(b));
    return r;
}

// Four bytes of E2M1 code pairs (one 32-bit word) -> four f16x2: byte j
// goes to o[j], its low nibble to the low half.  The word is split into its
// bytes with a vector mov so no shift/mask is spent per byte.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t* o) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}

// Binary32 -> E4M3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3(float s) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
    return r & 0xFFu;
}

// Two E4M3 bytes (low byte -> low half) -> f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    uint32_t r;
    uint16_t b = (uint16_t)two;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(b));
    return r;
}

__device__ __forceinline__ float e4m3_value(uint32_t byte) {
    uint32_t h = e4m3x2_to_f16x2(byte & 0xFFu);
    return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h) {
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// Two-lane binary32 arithmetic: one packed instruction, each lane rounded to
// nearest like the scalar add, subtract, multiply or fma.  The compiler has
// been seen to fuse a packed multiply into a packed add or subtract that
// consumes it (one rounding instead of two), .rn notwithstanding.  So every
// product that is summed later is formed as fma(x, y, z) with z = -0.0f read
// at run time (mulz2): exactly RN(x*y), and no single instruction can take
// its place together with the sum.  Products that only feed a conversion or
// another product stay plain multiplies (mul2).
#define BD_F32X2_OP(name, op)                                                                      \
    __device__ __forceinline__ float2 name(float2 a, float2 b) {                                   \
        float2 r;                                                                                  \
        asm("{\n\t.reg .b64 ra, rb, rr;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t" \
            op " rr, ra, rb;\n\tmov.b64 {%0, %1}, rr;\n\t}"                                     \
            : "=f"(r.x), "=f"(r.y)                                                                 \
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                             \
        return r;                                                                                  \
    }
BD_F32X2_OP(add2, "add.rn.f32x2")
BD_F32X2_OP(sub2, "sub.rn.f32x2")
BD_F32X2_OP(mul2, "mul.rn.f32x2")
#undef BD_F32X2_OP

// a * b + c per lane, rounded once.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{\n\t.reg .b64 ra, rb, rc, rr;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rr, ra, rb, rc;\n\tmov.b64 {%0, %1}, rr;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}
__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }
// a * b rounded once, for a product that a later add or subtract consumes;
// z holds a run-time -0.0f (the zero_addend of the kernel's arguments) in
// both lanes.
__device__ __forceinline__ float2 mulz2(float2 a, float2 b, float2 z) { return fma2(a, b, z); }

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

// Squared-error tree over 16 terms w[i] += w[i+8], then +4, +2, +1, with the
// terms held as pairs wp[i] = (w[2i], w[2i+1]): two additions per
// instruction until the last.
__device__ __forceinline__ float tree16x2(float2* wp) {
#pragma unroll
    for (int h = 4; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) wp[i] = add2(wp[i], wp[i + h]);
    return __fadd_rn(wp[0].x, wp[0].y);
}

// 2^e for e in [-127, 127], exact (2^-127 is subnormal).
__device__ __forceinline__ float pow2i(int e) {
    return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// The 8 code bytes of the 8 pairs quantized with exponent e (w0: elements
// 0-7, w1: 8-15) and their squared errors.
__device__ __forceinline__ void mx_enc_err16x2(const float2* xp, int e, float2 z, uint32_t& w0, uint32_t& w1,
                                               float2* wp) {
    const float2 down = splat2(pow2i(-e)), up = splat2(pow2i(e));
    w0 = 0;
    w1 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t hv;
        const float2 q = mul2(xp[i], down);
        const uint32_t byte = e2m1x2_enc_dec(q.x, q.y, hv);
        if (i < 4) w0 |= byte << (8 * i);
        else w1 |= byte << (8 * (i - 4));
        const float2 err = sub2(xp[i], mulz2(f16x2_to_float2(hv), up, z));
        wp[i] = mulz2(err, err, z);
    }
}

// floor(log2 a) for a finite a > 0 read from its exponent field.
__device__ __forceinline__ int ilog2f(float a) {
    uint32_t u = __float_as_uint(a);
    int e = (int)((u >> 23) & 0xFF);
    if (e != 0) return e - 127;
    return (31 - __clz((int)(u & 0x7FFFFF))) - 149;
}

// Order-preserving map of a non-NaN binary32 to u32 (a < b <=> key(a) <
// key(b)), so a float maximum can use the integer warp reduction; key(-inf)
// is 0x007FFFFF > 0, so key 0 is free to mean "no value".
__device__ __forceinline__ uint32_t f32_order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float f32_from_order_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// a / 6 correctly rounded.  For a >= 2^-100, Markstein's method for division
// by a constant: q0 = a * RN(1/6), the exact remainder r = a - 6 q0 by one
// FMA, and one more FMA q0 + r * RN(1/6) (valid while nothing underflows);
// smaller a takes the IEEE division.  Checked bit for bit against __fdiv_rn
// for every binary32 a in [0, 8] (the probability block maxima) by
// tests/div6_check.cu.
__device__ __forceinline__ float div6(float a) {
    if (a < 7.888609052210118e-31f) return __fdiv_rn(a, 6.0f);   // 2^-100
    const float y = 1.0f / 6.0f;
    const float q0 = __fmul_rn(a, y);
    const float r = __fmaf_rn(-q0, 6.0f, a);
    return __fmaf_rn(r, y, q0);
}

// The E4M3 scale byte of a / 6 for a probability block maximum a in [0, 8]:
// the same byte as e4m3(RN(a / 6)), without div6's branch (so the blocks of a
// page can be scheduled together).  For a >= 2^-100 the Markstein steps give
// RN(a / 6) itself; for smaller a they give a non-negative value below
// 2^-100, which rounds to the zero byte exactly as RN(a / 6) does (E4M3's
// smallest nonzero value is 2^-9).  Checked against e4m3(__fdiv_rn(a, 6)) for
// every binary32 a in [0, 8] by tests/div6_check.cu.
__device__ __forceinline__ uint32_t e4m3_div6(float a) {
    const float y = 1.0f / 6.0f;
    const float q0 = __fmul_rn(a, y);
    const float r = __fmaf_rn(-q0, 6.0f, a);
    return e4m3(__fmaf_rn(r, y, q0));
}

// ------------------------------------------------------------- f16x2 math --

// f16x2 of (2^klo, 2^khi) for k <= 0, by one conversion: 2^k is exact in
// binary32 down to 2^-126 (lower k clamped there), and its round-to-nearest
// f16 is 2^k itself down to 2^-24, 0 below (2^-25 is a tie, to the even 0) --
// the values f16_pow2 builds bit by bit.
__device__ __forceinline__ uint32_t f16x2_pow2(int klo, int khi) {
    const float lo = __uint_as_float((uint32_t)(max(klo, -126) + 127) << 23);
    const float hi = __uint_as_float((uint32_t)(max(khi, -126) + 127) << 23);
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// f16 bits of 2^k for k <= 0 (subnormal below -14, zero below -24).
__device__ __forceinline__ uint32_t f16_pow2(int k) {
    if (k >= -14) return (uint32_t)(k + 15) << 10;
    if (k >= -24) return 1u << (k + 24);
    return 0u;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t bcast_lo(uint32_t h) { return (h & 0xFFFFu) | (h << 16); }
__device__ __forceinline__ uint32_t bcast_hi(uint32_t h) { return (h >> 16) | (h & 0xFFFF0000u); }

// D += A(16x16, row) * B(16x8, col), f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------ mbarrier and TMA --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete, for at most
// limit_ns nanoseconds, giving up early when *abort_flag becomes nonzero.
// Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  const volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (abort_flag && *abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

// Bulk asynchronous copy global -> shared (TMA unit), completing `bytes`
// transaction bytes on the mbarrier.  Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 16-byte asynchronous copy global -> shared, cached in L2 only.  Both
// addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// L2 policy for data read exactly once: its lines are the first evicted, so
// a stream larger than L2 does not push out code or small reused data.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bulk_g2s with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Bulk prefetch of global memory into L2 (no shared-memory destination).
// Address 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void record_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ------------------------------------------ tensor memory and tcgen05 MMA --
//
// Fifth-generation tensor-core primitives (PTX tcgen05): tensor memory
// (TMEM, 128 lanes x 512 columns of 32 bits per SM) allocation, copies into
// it, block-scaled FP4 MMAs whose accumulators live there, and loads back to
// registers.  A TMEM address holds the lane in bits 31..16 and the column in
// bits 15..0; warp w of a warpgroup may load lanes 32 (w % 4) .. + 31 only.

// Allocate ncols (a power of two >= 32) columns; the base address is written
// to shared memory at dst.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// Free the allocation (the same warp that allocated; every tcgen05 operation
// on it must have completed).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Order tcgen05 operations against a thread synchronization (barrier or
// mbarrier) that precedes / follows them.
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, no swizzle: start address, the byte
// distance between core matrices (8 rows x 16 B) adjacent along K (lbo) and
// along M / N (sbo), and the descriptor version bit.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor of a block-scaled E2M1 x E2M1 MMA, both operands
// K-major, M = 128, N = n; ue8m0 selects UE8M0 scale factors (else UE4M3);
// sf_id picks the byte of each scale-factor word the MMA starts from.
__host__ __device__ constexpr uint32_t mma_idesc_e2m1(uint32_t n, bool ue8m0, uint32_t sf_id) {
    return (sf_id << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((ue8m0 ? 1u : 0u) << 23) |
           ((128u >> 4) << 24) | (sf_id << 29);
}

// D (tmem) = A x B^T (+ D if accumulate) with per-16-element UE4M3 scale
// factors (NVFP4) read from TMEM at sfa / sfb.  Issued by one thread.
__device__ __forceinline__ void mma_nvf4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
            "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}
// The same with per-32-element UE8M0 scale factors (MXFP4).
__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
            "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// Copy a 512-byte scale-factor group (32 lines of 16 B, contiguous in shared
// memory) into TMEM columns taddr .. taddr+3 of all four lane quarters: line i
// goes to lane 32 q + i of every quarter q.  Issued by the MMA thread; ordered
// before its later MMAs.
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint32_t smem_addr) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(smem_desc(smem_addr, 0, 128))
                 : "memory");
}

// Arrive on an mbarrier once every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Eight consecutive 32-bit columns of this thread's TMEM lane, then wait.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 lanes x 128 columns from the warp's lane quarter (starting at taddr),
// then wait: lane (g, t) = (lane / 4, lane % 4) receives, for j = 0..15,
// r[4 j + e] = (row g, column 8 j + 2 t + e) and r[4 j + 2 + e] = (row g + 8,
// column 8 j + 2 t + e), e = 0, 1 -- the accumulator layout of an m16n8 MMA.
__device__ __forceinline__ void tmem_ld_16x256b_x16(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Make this thread's generic shared-memory writes visible to the async proxy
// (bulk copies, tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace bd
