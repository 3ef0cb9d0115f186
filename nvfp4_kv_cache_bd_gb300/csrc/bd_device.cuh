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

// 2^e for e in [-127, 127], exact (2^-127 is subnormal).
__device__ __forceinline__ float pow2i(int e) {
    return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
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

// ------------------------------------------------------------- f16x2 math --

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

}  // namespace bd
