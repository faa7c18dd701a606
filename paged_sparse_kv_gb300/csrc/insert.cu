// insert.cu -- block-scaled quantize-and-insert into paged caches.
//
// FP8 (fp8_ds_mla record): vLLM deepseek_v41 ops, quantize_and_insert_k_cache;
// math of TokenSpeed deepseek_v4_ops.py, _fp8_ds_mla_cache_rows.
// MXFP4 (indexer keys): TokenSpeed deepseek_v4_ops.py,
// write_deepseek_v4_indexer_mxfp4_cache / read_deepseek_v4_indexer_mxfp4_cache.
//
// Design (HBM-bound scatter, no tensor cores):
//  * A group of LANES lanes owns one token row; each lane holds 16-byte chunks
//    (8 bf16) loaded with ld.global.nc.L1::no_allocate, so a 512-dim row is
//    two chunks per lane and one warp-wide load instruction moves 512 bytes.
//  * A quant block is 8 chunks (FP8, 64 dims) or 4 chunks (MXFP4, 32 dims),
//    held by 8 or 4 consecutive lanes: its amax is a 3- or 2-step
//    __shfl_xor reduction.
//  * amax is a 16-bit unsigned max over the bf16 magnitude bits, and the
//    scale exponent ceil(log2(amax / max_code)) is read off amax's own bits
//    (exact for bf16 amax; no divide, no log2); scaling is a packed
//    mul.rn.f32x2 per pair.
//  * Codes are packed with cvt.rn.satfinite.{e4m3x2,e2m1x2}.f32 and stored as
//    8-byte (FP8) / 4-byte (MXFP4) words: a group's stores of one record are
//    contiguous and coalesce; the rope tail moves as untouched 16-byte chunks.
//  * The scale bytes of a token are collected by shuffles into one lane and
//    written with a single aligned store.
//  * Each group handles UNROLL tokens with all loads issued before any use,
//    so enough bytes are in flight to cover HBM latency.
#include "insert.h"
#include "psk_common.cuh"

namespace psk {
namespace {

constexpr int kThreads = 256;

template <int NBYTES>
__device__ __forceinline__ void store_scale_word(uint8_t* p, uint64_t w) {
    if constexpr (NBYTES >= 8) {
        *reinterpret_cast<uint64_t*>(p) = w;
    } else if constexpr (NBYTES == 4) {
        *reinterpret_cast<uint32_t*>(p) = (uint32_t)w;
    } else if constexpr (NBYTES == 2) {
        *reinterpret_cast<uint16_t*>(p) = (uint16_t)w;
    } else {
        *p = (uint8_t)w;
    }
}

// Gather one byte per quant block (held by the first lane of each block's
// lane run) into the group's first lane and store the token's scale bytes.
// CHUNKS_PER_BLOCK lanes cover one block.
template <int LANES, int CPL, int CHUNKS_PER_BLOCK>
__device__ __forceinline__ void store_scale_bytes(const uint32_t (&sb)[CPL], unsigned gmask,
                                                  int grp, int gl, uint8_t* scl) {
    constexpr int NBLK = CPL * LANES / CHUNKS_PER_BLOCK;
    constexpr int WORD = NBLK < 8 ? NBLK : 8;
    uint64_t word = 0;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
#pragma unroll
        for (int kk = 0; kk < LANES / CHUNKS_PER_BLOCK; ++kk) {
            const uint32_t bv = __shfl_sync(gmask, sb[i], grp * LANES + kk * CHUNKS_PER_BLOCK);
            const int b = i * (LANES / CHUNKS_PER_BLOCK) + kk;
            word |= (uint64_t)(bv & 0xFFu) << (8 * (b % 8));
            if ((b % 8) == 7 || b == NBLK - 1) {
                if (gl == 0) store_scale_word<WORD>(scl + (b / 8) * 8, word);
                word = 0;
            }
        }
    }
}

template <int D, bool UE8M0, int UNROLL>
__global__ void __launch_bounds__(kThreads)
fp8_insert_kernel(const uint16_t* __restrict__ k, int64_t k_row_stride,
                  const int64_t* __restrict__ slots, int64_t n,
                  uint8_t* __restrict__ cache, int64_t capacity, int64_t page_stride,
                  int32_t bs, int32_t shift, int32_t rope, int32_t* __restrict__ err) {
    constexpr int CHUNKS = D / 8;
    constexpr int LANES = CHUNKS < kWarp ? CHUNKS : kWarp;
    constexpr int CPL = CHUNKS / LANES;
    constexpr int NBLK = D / 64;
    constexpr int SDIM = UE8M0 ? NBLK : 4 * NBLK;

    const int lane = threadIdx.x & 31;
    const int grp = lane / LANES, gl = lane % LANES;
    const unsigned gmask =
        LANES == 32 ? 0xFFFFFFFFu : (((1u << LANES) - 1u) << (grp * LANES));
    const int64_t gid = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / LANES;
    const int64_t tok0 = gid * UNROLL;
    const int nope = D - rope;
    const int64_t ts = nope + 2 * rope;
    pdl_wait();
    pdl_launch_dependents();

    uint4 v[UNROLL][CPL];
    int64_t s[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const int64_t t = tok0 + u;
        s[u] = -1;
        if (t < n) {
            s[u] = __ldg(slots + t);
            const uint16_t* row = k + t * k_row_stride;
#pragma unroll
            for (int i = 0; i < CPL; ++i) v[u][i] = ld_stream_v4(row + 8 * (gl + i * LANES));
        }
    }

#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const int64_t sl = s[u];
        if (sl < 0) continue;  // same token for the whole group: uniform
        if (sl >= capacity) {
            if (gl == 0 && err) atomicAdd(err, 1);
            continue;
        }
        int64_t off;
        const int64_t page = div_block(sl, bs, shift, off);
        uint8_t* base = cache + page * page_stride;
        uint8_t* data = base + off * ts;
        uint8_t* scl = base + (int64_t)bs * ts + off * SDIM;

        uint32_t sb[CPL];
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int c = gl + i * LANES;
            const uint4 w = v[u][i];
            float x[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                          bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
            uint32_t amb = absmax_bf16x8_bits(w);
            amb = max(amb, __shfl_xor_sync(gmask, amb, 1));
            amb = max(amb, __shfl_xor_sync(gmask, amb, 2));
            amb = max(amb, __shfl_xor_sync(gmask, amb, 4));
            const float am = __uint_as_float(amb << 16);
            if (8 * c < nope) {  // uniform over the block's 8 lanes
                float y[8];
                if constexpr (UE8M0) {
                    const float a = fmaxf(am, 1.0e-4f);
                    const int e = ceil_log2_div_const(a, 0x600000u, 8);  // / 448
                    const int b = min(max(e + 127, 0), 255);
                    const uint64_t pw2 = splat_f32x2(exp2_int(-e));
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {
                        y[j] = x[j];
                        y[j + 1] = x[j + 1];
                        mul2_rn(y[j], y[j + 1], pw2);
                        y[j] = clamp_sym(y[j], 448.0f);
                        y[j + 1] = clamp_sym(y[j + 1], 448.0f);
                    }
                    sb[i] = (uint32_t)b;
                } else {
                    const float a = fmaxf(am, 1.0e-12f);
                    const float sc = __fdiv_rn(a, 448.0f);
#pragma unroll
                    for (int j = 0; j < 8; ++j) y[j] = clamp_sym(__fdiv_rn(x[j], sc), 448.0f);
                    sb[i] = __float_as_uint(sc);
                }
                uint2 q;
                q.x = cvt_e4m3x2(y[0], y[1]) | (cvt_e4m3x2(y[2], y[3]) << 16);
                q.y = cvt_e4m3x2(y[4], y[5]) | (cvt_e4m3x2(y[6], y[7]) << 16);
                st_v2(data + 8 * c, q);
            } else {
                st_v4(data + 16 * c - nope, w);  // rope tail: bf16 verbatim
                sb[i] = 0;
            }
        }
        if constexpr (UE8M0) {
            store_scale_bytes<LANES, CPL, 8>(sb, gmask, grp, gl, scl);
        } else {
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int c = gl + i * LANES;
                if ((c & 7) == 0) *reinterpret_cast<uint32_t*>(scl + 4 * (c / 8)) = sb[i];
            }
        }
    }
}

// Lanes per token of the MXFP4 insert: two 16-byte chunks per lane where the
// row allows it (halving the per-token slot, address and branch work of one
// chunk per lane), at least the 4 lanes of one 32-element block.
template <int D>
__host__ __device__ constexpr int mxfp4_lanes() {
    constexpr int half = D / 16;
    return half < 4 ? 4 : (half > kWarp ? kWarp : half);
}

template <int D, int UNROLL>
__global__ void __launch_bounds__(kThreads)
mxfp4_insert_kernel(const uint16_t* __restrict__ k, int64_t k_row_stride,
                    const int64_t* __restrict__ slots, int64_t n,
                    uint8_t* __restrict__ cache, int64_t capacity, int64_t page_stride,
                    int32_t bs, int32_t shift, int32_t* __restrict__ err) {
    constexpr int CHUNKS = D / 8;
    constexpr int LANES = mxfp4_lanes<D>();
    constexpr int CPL = CHUNKS / LANES;
    constexpr int VB = D / 2;   // value bytes per token
    static_assert(CPL * LANES == CHUNKS && LANES % 4 == 0, "a block spans 4 lanes");

    const int lane = threadIdx.x & 31;
    const int grp = lane / LANES, gl = lane % LANES;
    const unsigned gmask =
        LANES == 32 ? 0xFFFFFFFFu : (((1u << LANES) - 1u) << (grp * LANES));
    const int64_t gid = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / LANES;
    const int64_t tok0 = gid * UNROLL;
    pdl_wait();
    pdl_launch_dependents();

    uint4 v[UNROLL][CPL];
    int64_t s[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const int64_t t = tok0 + u;
        s[u] = -1;
        if (t < n) {
            s[u] = __ldg(slots + t);
            const uint16_t* row = k + t * k_row_stride;
#pragma unroll
            for (int i = 0; i < CPL; ++i) v[u][i] = ld_stream_v4(row + 8 * (gl + i * LANES));
        }
    }

#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const int64_t sl = s[u];
        if (sl < 0) continue;
        if (sl >= capacity) {
            if (gl == 0 && err) atomicAdd(err, 1);
            continue;
        }
        int64_t off;
        const int64_t page = div_block(sl, bs, shift, off);
        uint8_t* base = cache + page * page_stride;
        uint8_t* vals = base + off * VB;
        uint8_t* scl = base + (int64_t)bs * VB + off * (D / 32);

#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int c = gl + i * LANES;
            const uint4 w = v[u][i];
            float x[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                          bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
            uint32_t amb = absmax_bf16x8_bits(w);
            amb = max(amb, __shfl_xor_sync(gmask, amb, 1));
            amb = max(amb, __shfl_xor_sync(gmask, amb, 2));
            const float a = fmaxf(__uint_as_float(amb << 16), 1.0e-4f);
            const int e = ceil_log2_div_const(a, 0x400000u, 2);  // / 6
            const uint64_t pw2 = splat_f32x2(exp2_int(-e));
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float lo = x[2 * j], hi = x[2 * j + 1];
                mul2_rn(lo, hi, pw2);
                word |= (cvt_e2m1x2(lo, hi) & 0xFFu) << (8 * j);
            }
            *reinterpret_cast<uint32_t*>(vals + 4 * c) = word;
            // the block's first lane writes its scale byte
            if ((gl & 3) == 0) scl[c / 4] = (uint8_t)min(max(e + 127, 0), 254);
        }
    }
}

// ---- FP8 indexer record --------------------------------------------------------------
//
// TokenSpeed write_deepseek_v4_indexer_fp8_cache (the "[values | fp32 scale]"
// page layout) with the rule of _fp8_e4m3_pow2_bytes: one power-of-two
// binary32 scale per token, 2^ceil(log2(max(amax / 448, 1e-10))) -- the
// quotient is floored, not amax -- and codes e4m3(x / scale), computed as
// x * 2^-e (the same single rounding of the same exact value).  Lanes as the
// MXFP4 insert; the row amax is an integer shuffle-max over the token's lanes.
template <int D, int UNROLL>
__global__ void __launch_bounds__(kThreads)
fp8_indexer_insert_kernel(const uint16_t* __restrict__ k, int64_t k_row_stride,
                          const int64_t* __restrict__ slots, int64_t n,
                          uint8_t* __restrict__ cache, int64_t capacity, int64_t page_stride,
                          int32_t bs, int32_t shift, int32_t* __restrict__ err) {
    constexpr int CHUNKS = D / 8;
    constexpr int LANES = mxfp4_lanes<D>();
    constexpr int CPL = CHUNKS / LANES;
    static_assert(CPL * LANES == CHUNKS, "whole chunks per lane");

    const int lane = threadIdx.x & 31;
    const int grp = lane / LANES, gl = lane % LANES;
    const unsigned gmask =
        LANES == 32 ? 0xFFFFFFFFu : (((1u << LANES) - 1u) << (grp * LANES));
    const int64_t gid = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / LANES;
    const int64_t tok0 = gid * UNROLL;
    pdl_wait();
    pdl_launch_dependents();

    uint4 v[UNROLL][CPL];
    int64_t s[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const int64_t t = tok0 + u;
        s[u] = -1;
        if (t < n) {
            s[u] = __ldg(slots + t);
            const uint16_t* row = k + t * k_row_stride;
#pragma unroll
            for (int i = 0; i < CPL; ++i) v[u][i] = ld_stream_v4(row + 8 * (gl + i * LANES));
        }
    }

#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const int64_t sl = s[u];
        if (sl < 0) continue;
        if (sl >= capacity) {
            if (gl == 0 && err) atomicAdd(err, 1);
            continue;
        }
        int64_t off;
        const int64_t page = div_block(sl, bs, shift, off);
        uint8_t* base = cache + page * page_stride;
        uint8_t* vals = base + off * D;

        uint32_t amb = 0;
#pragma unroll
        for (int i = 0; i < CPL; ++i) amb = max(amb, absmax_bf16x8_bits(v[u][i]));
#pragma unroll
        for (int m = 1; m < LANES; m <<= 1) amb = max(amb, __shfl_xor_sync(gmask, amb, m));
        const float q = fmaxf(__fdiv_rn(__uint_as_float(amb << 16), 448.0f), 1.0e-10f);
        const int e = ceil_log2_pos(q);
        const uint64_t pw2 = splat_f32x2(exp2_int(-e));
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int c = gl + i * LANES;
            const uint4 w = v[u][i];
            float x[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                          bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
            for (int j = 0; j < 8; j += 2) mul2_rn(x[j], x[j + 1], pw2);
            uint2 q8;
            q8.x = cvt_e4m3x2(x[0], x[1]) | (cvt_e4m3x2(x[2], x[3]) << 16);
            q8.y = cvt_e4m3x2(x[4], x[5]) | (cvt_e4m3x2(x[6], x[7]) << 16);
            st_v2(vals + 8 * c, q8);
        }
        if (gl == 0)
            *reinterpret_cast<float*>(base + (int64_t)bs * D + off * 4) = exp2_int(e);
    }
}

// ---- indexer_k_norm_rope_store ---------------------------------------------------------
//
// vLLM deepseek_v41 ops, indexer_k_norm_rope_store: k_norm -> RoPE -> quant ->
// paged store of 128-dim indexer keys.  One warp per token; lane l holds dims
// 4l..4l+3 (one 8-byte load).
//  * Emission: slot >= 0 and the token closes its compress group,
//    (pos + 1) % ratio == 0 (TokenSpeed _compress_v4_state_windows_capturable's
//    valid_token rule).
//  * RMSNorm in binary32, every operation rounded once (no contraction): the
//    sum of squares is a pairwise sum -- (s0 + s1) + (s2 + s3) in the lane,
//    then xor-shuffles over 1, 2, 4, 8, 16 lanes, i.e. recursive halving of
//    the index range; variance = sum / 128; r = binary32 of 1 / sqrt(variance
//    + eps) with the square root and the quotient in IEEE binary64;
//    y = (x * r) * weight.
//  * GPT-J RoPE (TokenSpeed _apply_gptj_rope_tail_rows) on dims 64..127 (lanes
//    16..31: two pairs each) at the cos_sin row of the group's first position
//    floor(pos / ratio) * ratio.
//  * MXFP4 record (8-lane blocks) or FP8 indexer record (row amax), with the
//    inserts' rules.
template <bool FP4>
__global__ void __launch_bounds__(kThreads) norm_rope_store_kernel(NormRopeParams p,
                                                                   int32_t shift) {
    const int lane = threadIdx.x & 31;
    const int64_t t = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / kWarp;
    pdl_wait();
    pdl_launch_dependents();
    if (t >= p.num_tokens) return;
    const int64_t sl = __ldg(p.slots + t);
    if (sl < 0) return;
    const int64_t pos = __ldg(p.positions + t);
    int64_t rem = (pos + 1) % p.ratio;
    if (rem < 0) rem += p.ratio;
    if (rem != 0) return;  // not a group boundary: the row is not read
    int64_t grp = pos / p.ratio;
    if (pos % p.ratio != 0 && pos < 0) grp -= 1;
    const int64_t prow = grp * p.ratio;
    const int64_t capacity = p.num_pages * (int64_t)p.block_size;
    if (sl >= capacity || prow < 0 || prow >= p.max_pos) {
        if (lane == 0 && p.err_count) atomicAdd(p.err_count, 1);
        return;
    }

    const uint2 kw = ld_nc_v2(p.k + t * p.k_row_stride + 4 * lane);
    float y[4] = {bf16_lo(kw.x), bf16_hi(kw.x), bf16_lo(kw.y), bf16_hi(kw.y)};
    float ss = __fadd_rn(__fadd_rn(__fmul_rn(y[0], y[0]), __fmul_rn(y[1], y[1])),
                         __fadd_rn(__fmul_rn(y[2], y[2]), __fmul_rn(y[3], y[3])));
#pragma unroll
    for (int m = 1; m < kWarp; m <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, m));
    const float variance = __fdiv_rn(ss, 128.0f);
    const float r =
        __double2float_rn(__ddiv_rn(1.0, __dsqrt_rn((double)__fadd_rn(variance, p.eps))));
    const float4 wv = __ldg(reinterpret_cast<const float4*>(p.weight) + lane);
    y[0] = __fmul_rn(__fmul_rn(y[0], r), wv.x);
    y[1] = __fmul_rn(__fmul_rn(y[1], r), wv.y);
    y[2] = __fmul_rn(__fmul_rn(y[2], r), wv.z);
    y[3] = __fmul_rn(__fmul_rn(y[3], r), wv.w);
    if (lane >= 16) {
        const float* cs = p.cos_sin + prow * p.cs_stride;
        const int i0 = 2 * lane - 32;  // pair index of dims 4l, 4l + 1
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float c = __ldg(cs + i0 + h), sn = __ldg(cs + 32 + i0 + h);
            const float e = y[2 * h], o = y[2 * h + 1];
            y[2 * h] = __fsub_rn(__fmul_rn(e, c), __fmul_rn(o, sn));
            y[2 * h + 1] = __fadd_rn(__fmul_rn(e, sn), __fmul_rn(o, c));
        }
    }

    int64_t off;
    const int64_t page = div_block(sl, p.block_size, shift, off);
    uint8_t* base = p.cache + page * p.page_stride;
    float a = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
    if constexpr (FP4) {
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, m));
        const int e = ceil_log2_pos(__fdiv_rn(fmaxf(a, 1.0e-4f), 6.0f));
        const float pw = exp2_int(-e);
        const uint32_t lo = cvt_e2m1x2(__fmul_rn(y[0], pw), __fmul_rn(y[1], pw)) & 0xFFu;
        const uint32_t hi = cvt_e2m1x2(__fmul_rn(y[2], pw), __fmul_rn(y[3], pw)) & 0xFFu;
        *reinterpret_cast<uint16_t*>(base + off * 64 + 2 * lane) = (uint16_t)(lo | (hi << 8));
        if ((lane & 7) == 0)
            base[(int64_t)p.block_size * 64 + off * 4 + lane / 8] =
                (uint8_t)min(max(e + 127, 0), 254);
    } else {
#pragma unroll
        for (int m = 1; m < kWarp; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, m));
        const int e = ceil_log2_pos(fmaxf(__fdiv_rn(a, 448.0f), 1.0e-10f));
        const float pw = exp2_int(-e);
        const uint32_t q = cvt_e4m3x2(__fmul_rn(y[0], pw), __fmul_rn(y[1], pw)) |
                           (cvt_e4m3x2(__fmul_rn(y[2], pw), __fmul_rn(y[3], pw)) << 16);
        *reinterpret_cast<uint32_t*>(base + off * 128 + 4 * lane) = q;
        if (lane == 0)
            *reinterpret_cast<float*>(base + (int64_t)p.block_size * 128 + off * 4) = exp2_int(e);
    }
}

template <int D, bool UE8M0>
cudaError_t fp8_insert_dispatch(const InsertParams& p, cudaStream_t stream) {
    constexpr int UNROLL = 2;
    constexpr int LANES = (D / 8) < kWarp ? (D / 8) : kWarp;
    const int64_t groups = (p.num_tokens + UNROLL - 1) / UNROLL;
    const int64_t threads = groups * LANES;
    const int64_t blocks = (threads + kThreads - 1) / kThreads;
    return launch_pdl(fp8_insert_kernel<D, UE8M0, UNROLL>, dim3((unsigned)blocks), dim3(kThreads),
                      0, stream, static_cast<const uint16_t*>(p.k), p.k_row_stride, p.slots,
                      p.num_tokens, p.cache, p.num_pages * (int64_t)p.block_size,
                      p.page_stride, p.block_size, log2_if_pow2(p.block_size), p.rope_dim,
                      p.err_count);
}

template <int D>
cudaError_t mxfp4_insert_dispatch(const InsertParams& p, cudaStream_t stream) {
    constexpr int UNROLL = 2;
    constexpr int LANES = mxfp4_lanes<D>();
    const int64_t groups = (p.num_tokens + UNROLL - 1) / UNROLL;
    const int64_t threads = groups * LANES;
    const int64_t blocks = (threads + kThreads - 1) / kThreads;
    return launch_pdl(mxfp4_insert_kernel<D, UNROLL>, dim3((unsigned)blocks), dim3(kThreads), 0,
                      stream, static_cast<const uint16_t*>(p.k), p.k_row_stride, p.slots,
                      p.num_tokens, p.cache, p.num_pages * (int64_t)p.block_size,
                      p.page_stride, p.block_size, log2_if_pow2(p.block_size), p.err_count);
}

template <int D>
cudaError_t fp8_indexer_insert_dispatch(const InsertParams& p, cudaStream_t stream) {
    constexpr int UNROLL = 2;
    constexpr int LANES = mxfp4_lanes<D>();
    const int64_t groups = (p.num_tokens + UNROLL - 1) / UNROLL;
    const int64_t threads = groups * LANES;
    const int64_t blocks = (threads + kThreads - 1) / kThreads;
    return launch_pdl(fp8_indexer_insert_kernel<D, UNROLL>, dim3((unsigned)blocks),
                      dim3(kThreads), 0, stream, static_cast<const uint16_t*>(p.k),
                      p.k_row_stride, p.slots, p.num_tokens, p.cache,
                      p.num_pages * (int64_t)p.block_size, p.page_stride, p.block_size,
                      log2_if_pow2(p.block_size), p.err_count);
}

}  // namespace

cudaError_t launch_fp8_indexer_insert(const InsertParams& p, cudaStream_t stream) {
    switch (p.head_dim) {
        case 32: return fp8_indexer_insert_dispatch<32>(p, stream);
        case 64: return fp8_indexer_insert_dispatch<64>(p, stream);
        case 128: return fp8_indexer_insert_dispatch<128>(p, stream);
        case 256: return fp8_indexer_insert_dispatch<256>(p, stream);
        case 512: return fp8_indexer_insert_dispatch<512>(p, stream);
        case 1024: return fp8_indexer_insert_dispatch<1024>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_norm_rope_store(const NormRopeParams& p, cudaStream_t stream) {
    const int64_t blocks = (p.num_tokens * kWarp + kThreads - 1) / kThreads;
    const int32_t shift = log2_if_pow2(p.block_size);
    auto kern = p.record == 1 ? norm_rope_store_kernel<true> : norm_rope_store_kernel<false>;
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), 0, stream, p, shift);
}

cudaError_t launch_fp8_insert(const InsertParams& p, cudaStream_t stream) {
    const bool ue = p.is_ue8m0 != 0;
    switch (p.head_dim) {
        case 64: return ue ? fp8_insert_dispatch<64, true>(p, stream) : fp8_insert_dispatch<64, false>(p, stream);
        case 128: return ue ? fp8_insert_dispatch<128, true>(p, stream) : fp8_insert_dispatch<128, false>(p, stream);
        case 256: return ue ? fp8_insert_dispatch<256, true>(p, stream) : fp8_insert_dispatch<256, false>(p, stream);
        case 512: return ue ? fp8_insert_dispatch<512, true>(p, stream) : fp8_insert_dispatch<512, false>(p, stream);
        case 1024: return ue ? fp8_insert_dispatch<1024, true>(p, stream) : fp8_insert_dispatch<1024, false>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_mxfp4_insert(const InsertParams& p, cudaStream_t stream) {
    switch (p.head_dim) {
        case 32: return mxfp4_insert_dispatch<32>(p, stream);
        case 64: return mxfp4_insert_dispatch<64>(p, stream);
        case 128: return mxfp4_insert_dispatch<128>(p, stream);
        case 256: return mxfp4_insert_dispatch<256>(p, stream);
        case 512: return mxfp4_insert_dispatch<512>(p, stream);
        case 1024: return mxfp4_insert_dispatch<1024>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace psk
