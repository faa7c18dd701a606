// psk_common.cuh -- device helpers shared by the libpsk kernels (sm_103a).
//
// Conversions go through the PTX `cvt` forms for FP8/FP4 (round to nearest
// even, satfinite) and bf16; exponent work is done on binary32 bit patterns.
// Build without --use_fast_math: every product and quotient here must be the
// IEEE-rounded one, with subnormals kept.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace psk {

constexpr int kWarp = 32;

// ---- memory ----------------------------------------------------------------

// 16-byte read-only load that does not allocate in L1 (rows read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ld_nc_v2(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_nc_u8(const void* p) {
    uint16_t r;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// Streaming (evict-first) stores for outputs that are not re-read here.
__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// 32 bytes of streaming output at p: one 256-bit store when `v8` (p 32-byte
// aligned; a warp storing 32 consecutive chunks covers 1 KB, which this part
// writes at ~7.2 TB/s against ~6.5 TB/s for 16-byte stores), else two 16-byte
// stores.
__device__ __forceinline__ void store_out32(void* p, uint4 lo, uint4 hi, int v8) {
    if (v8) {
        asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                     :: "l"(p), "r"(lo.x), "r"(lo.y), "r"(lo.z), "r"(lo.w), "r"(hi.x), "r"(hi.y),
                        "r"(hi.z), "r"(hi.w) : "memory");
    } else {
        st_stream_v4(p, lo);
        st_stream_v4(static_cast<uint8_t*>(p) + 16, hi);
    }
}

__device__ __forceinline__ void st_v2(void* p, uint2 v) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// ---- bf16 / binary32 ----------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two binary32 -> packed bf16x2 (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 2^k as binary32 for k in [-149, 128] (k = 128 gives +inf).
__device__ __forceinline__ float exp2_int(int k) {
    if (k >= -126) return __uint_as_float((uint32_t)(k + 127) << 23);
    return __uint_as_float(1u << (k + 149));
}

// The factor f with x * f == x / scale for a power-of-two binary32 scale
// 2^e, e in [-127, 128]: 2^-e while 2^e is finite (both a single rounding of
// the same exact value); at e = 128 the scale itself rounds to +inf, and
// x / inf (+-0 for finite x, NaN for +-inf and NaN) is x * 0.
__device__ __forceinline__ float inv_pow2_scale(int e) { return e >= 128 ? 0.0f : exp2_int(-e); }

// Smallest e with 2^e >= q for finite q > 0 (normal q): read off the bits.
// q = +inf gives 128.
__device__ __forceinline__ int ceil_log2_pos(float q) {
    const uint32_t b = __float_as_uint(q);
    const int e = (int)((b >> 23) & 0xFFu) - 127;
    return e + ((b & 0x7FFFFFu) != 0u ? 1 : 0);
}

// ceil(log2(RN(a / c))) for c = cs * 2^cx with significand cs (mantissa bits
// cs_mant), without dividing.  Write a = s * 2^x, s in [1, 2).  Then
// a / c <= 2^k  <=>  s <= cs * 2^(k + cx - x), so the exact answer is
// x - cx + (s > cs).  It equals the answer for the rounded quotient RN(a / c)
// whenever a / c is either exactly a power of two or farther than half an ulp
// from every power of two.  For c = 448 = 1.75 * 2^8 and c = 6 = 1.5 * 2^2 that
// holds for every a with an 8-bit significand (a bf16 block amax: a / c is a
// power of two exactly when s = cs, and otherwise at least ~0.4% away), for
// the 1e-4 floor, and for every normal binary32 a: the significands next to
// cs are cs +- 2^-23, whose quotients s / cs lie at least 2^-23 / 1.75 above 1
// (more than the half ulp 2^-24 above 1) or below 1 (more than the half ulp
// 2^-25 below 1), so RN(a / c) is a power of two exactly when s = cs and is
// on the same side of it as a / c otherwise (the quotient must stay normal).
// a must be positive and normal; +inf gives 128 (as the quotient inf would).
__device__ __forceinline__ int ceil_log2_div_const(float a, uint32_t cs_mant, int cx) {
    const uint32_t b = __float_as_uint(a);
    if (b >= 0x7F800000u) return 128;
    const int x = (int)(b >> 23) - 127;
    return x - cx + ((b & 0x7FFFFFu) > cs_mant ? 1 : 0);
}

// Elementwise max of two bf16x2 words.  max.bf16x2 (no .NaN) returns the
// other operand where one is NaN and NaN only where both are.
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Per-half largest |x| of eight bf16 values (packed in a uint4), as a bf16x2
// word: NaN entries are passed over, as an ordered "a > amax" scan does.
__device__ __forceinline__ uint32_t absmax_bf16x8_pair(uint4 w) {
    constexpr uint32_t M = 0x7FFF7FFFu;
    return bmax2(bmax2(w.x & M, w.y & M), bmax2(w.z & M, w.w & M));
}

// The same over a whole bf16x2 word, as a binary32 (exact).
__device__ __forceinline__ float absmax_of_pair(uint32_t m) { return fmaxf(bf16_lo(m), bf16_hi(m)); }

// Largest |x| of eight bf16 values (packed in a uint4) as a binary32 max tree
// (exact); fmaxf passes over NaN like max.bf16x2.  Cheaper than the packed
// form where the kernel unpacks the values anyway.
__device__ __forceinline__ float absmax_bf16x8(uint4 w) {
    return fmaxf(fmaxf(fmaxf(fabsf(bf16_lo(w.x)), fabsf(bf16_hi(w.x))),
                       fmaxf(fabsf(bf16_lo(w.y)), fabsf(bf16_hi(w.y)))),
                 fmaxf(fmaxf(fabsf(bf16_lo(w.z)), fabsf(bf16_hi(w.z))),
                       fmaxf(fabsf(bf16_lo(w.w)), fabsf(bf16_hi(w.w)))));
}

// {lo, hi} * {s, s} in one packed multiply (IEEE RN per element, no flush).
__device__ __forceinline__ void mul2_rn(float& lo, float& hi, uint64_t s2) {
    asm("{\n\t.reg .b64 x, y;\n\t"
        "mov.b64 x, {%0, %1};\n\t"
        "mul.rn.f32x2 y, x, %2;\n\t"
        "mov.b64 {%0, %1}, y;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "l"(s2));
}

// Decode of a UE8M0 byte: 2^(b - 127) as binary32 (b = 255 -> +inf).
__device__ __forceinline__ float ue8m0_scale(uint32_t b) {
    return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// ---- FP8 E4M3 / FP4 E2M1 --------------------------------------------------------

// Two binary32 -> two E4M3 bytes (lo in bits 0..7), RNE, satfinite.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two binary32 -> two E2M1 nibbles (lo in bits 0..3), RNE, satfinite.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u16.u8 %0, t;\n\t}"
        : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two E4M3 bytes (bits 0..15) -> f16x2, exact.
__device__ __forceinline__ uint32_t cvt_e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t r;
    const uint16_t in = (uint16_t)two_bytes;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(in));
    return r;
}

// Two E2M1 nibbles (bits 0..7) -> f16x2, exact.
__device__ __forceinline__ uint32_t cvt_e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    const uint16_t in = (uint16_t)byte;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.u8.u16 t, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(r) : "h"(in));
    return r;
}

__device__ __forceinline__ float f16_lo(uint32_t h2) {
    float f;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(h2));
    return f;
}

__device__ __forceinline__ float f16_hi(uint32_t h2) {
    float f;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(h2));
    return f;
}

// Two f16 (packed) times a binary32 scale pair {s, s}, rounded to packed bf16:
// each half widened to binary32 exactly, one packed multiply (mul.rn.f32x2,
// IEEE round-to-nearest per element, subnormals kept), then cvt.rn.bf16x2.
__device__ __forceinline__ uint32_t scale_f16x2_to_bf16x2(uint32_t h2, uint64_t s2) {
    const float lo = f16_lo(h2), hi = f16_hi(h2);
    uint32_t r;
    asm("{\n\t.reg .b64 x, y;\n\t.reg .b32 a, b;\n\t"
        "mov.b64 x, {%1, %2};\n\t"
        "mul.rn.f32x2 y, x, %3;\n\t"
        "mov.b64 {a, b}, y;\n\t"
        "cvt.rn.bf16x2.f32 %0, b, a;\n\t}"
        : "=r"(r)
        : "f"(lo), "f"(hi), "l"(s2));
    return r;
}

__device__ __forceinline__ uint64_t splat_f32x2(float s) {
    const uint64_t b = __float_as_uint(s);
    return (b << 32) | b;
}

// ---- programmatic dependent launch ------------------------------------------------
//
// Every libpsk kernel is launched with programmatic stream serialisation, so
// it may start while the previous kernel on the stream is still finishing.
// pdl_wait() blocks until that kernel has completed and its writes are
// visible; every kernel calls it before its first global-memory access.
// pdl_launch_dependents() lets the next kernel on the stream begin launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- integer helpers ---------------------------------------------------------------

__host__ __device__ __forceinline__ int log2_if_pow2(int x) {
    if (x <= 0 || (x & (x - 1))) return -1;
    int s = 0;
    while ((1 << s) < x) ++s;
    return s;
}

// Quotient and remainder of v >= 0 by a page's block size bs.  shift =
// log2_if_pow2(bs), computed once on the host: a shift and a mask when bs is
// a power of two, else a 32-bit divide while v fits in 32 bits, else a 64-bit
// one (an emulated 64-bit divide costs dozens of instructions per call).
__device__ __forceinline__ int64_t div_block(int64_t v, int32_t bs, int32_t shift, int64_t& rem) {
    if (shift >= 0) {
        rem = v & (int64_t)(bs - 1);
        return v >> shift;
    }
    if ((uint64_t)v <= 0xFFFFFFFFull) {
        const uint32_t q = (uint32_t)v / (uint32_t)bs;
        rem = (int64_t)((uint32_t)v - q * (uint32_t)bs);
        return (int64_t)q;
    }
    const int64_t q = v / bs;
    rem = v - q * bs;
    return q;
}

__device__ __forceinline__ int32_t div_block32(int32_t v, int32_t bs, int32_t shift, int32_t& rem) {
    if (shift >= 0) {
        rem = v & (bs - 1);
        return v >> shift;
    }
    const uint32_t q = (uint32_t)v / (uint32_t)bs;
    rem = (int32_t)((uint32_t)v - q * (uint32_t)bs);
    return (int32_t)q;
}

}  // namespace psk

// ---- mbarrier + bulk async copy (TMA, non-tensor) ----------------------------------

namespace psk {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One try_wait; the thread may be suspended in hardware (up to the hint, in
// ns) until the phase completes, so a waiting warp does not spin on issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the barrier phase with the given parity; gives up after
// `limit_ns` of wall time and returns false (the caller records the timeout).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint2 lds_v2(const void* p) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(smem_u32(p)));
    return r;
}

__device__ __forceinline__ uint4 lds_v4(const void* p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(smem_u32(p)));
    return r;
}

__device__ __forceinline__ uint32_t lds_u8(const void* p) {
    uint16_t r;
    asm volatile("ld.shared.u8 %0, [%1];" : "=h"(r) : "r"(smem_u32(p)));
    return r;
}

__device__ __forceinline__ uint32_t lds_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(smem_u32(p)));
    return r;
}

}  // namespace psk
