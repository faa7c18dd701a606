// insert.cu -- block-scaled quantize-and-insert into paged caches.
//
// FP8 (fp8_ds_mla record): vLLM deepseek_v41 ops, quantize_and_insert_k_cache;
// math of TokenSpeed deepseek_v4_ops.py, _fp8_ds_mla_cache_rows.
// MXFP4 (indexer keys): TokenSpeed deepseek_v4_ops.py,
// write_deepseek_v4_indexer_mxfp4_cache / read_deepseek_v4_indexer_mxfp4_cache.
//
// Design (HBM-bound scatter, no tensor cores):
//  * A group of LANES lanes owns one token row; each lane holds 16-byte chunks
//    (8 bf16) loaded through the read-only path, so a 512-dim row is two
//    chunks per lane and one warp-wide load instruction moves 512 bytes.
//  * A quant block is 8 chunks (FP8, 64 dims) or 4 chunks (MXFP4, 32 dims).
//    FP8: 8 consecutive lanes, one chunk each, a 3-step __shfl_xor reduction.
//    MXFP4: each lane holds adjacent chunks, so the block spans fewer lanes.
//  * amax is exact and passes over NaN, as the oracle's ordered scan does: a
//    binary32 max tree of the magnitudes (FP8, MXFP4) or a packed max.bf16x2
//    (FP8 indexer: measured faster there), then shuffles across lanes.  The
//    scale exponent ceil(log2(amax / max_code)) is read off amax's own bits
//    (no divide, no log2); scaling is a packed mul.rn.f32x2 per pair.
//  * Codes are packed with cvt.rn.satfinite.{e4m3x2,e2m1x2}.f32 and stored as
//    8-byte words (FP8: one per chunk; MXFP4: a lane's adjacent chunks at 128
//    dims): a group's stores of one record are contiguous and coalesce; the
//    rope tail moves as untouched 16-byte chunks.
//  * Each quant block's first lane stores the block's scale byte (or binary32
//    scale): the bytes of one token are adjacent, so the stores of a group
//    coalesce into one request per chunk column.
//  * Each group handles UNROLL tokens with all loads issued before any use
//    (two for the MXFP4 and indexer inserts; one for the FP8 insert, whose
//    32-register build keeps 64 warps per SM in flight instead).
#include "insert.h"
#include "psk_common.cuh"

namespace psk {
namespace {

constexpr int kThreads = 256;

// Blocks of the FP8 insert resident per SM: 8 (32 registers, no spills, 64
// warps each with one token's loads in flight) up to 512 dims; wider rows hold
// four chunks per lane and would spill at 32 registers.
template <int D>
constexpr int fp8_insert_min_blocks() { return D <= 512 ? 8 : 1; }

template <int D, bool UE8M0, int UNROLL>
__global__ void __launch_bounds__(kThreads, fp8_insert_min_blocks<D>())
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

#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int c = gl + i * LANES;
            const uint4 w = v[u][i];
            float x[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                          bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
            float am = absmax_bf16x8(w);
            am = fmaxf(am, __shfl_xor_sync(gmask, am, 1));
            am = fmaxf(am, __shfl_xor_sync(gmask, am, 2));
            am = fmaxf(am, __shfl_xor_sync(gmask, am, 4));
            const bool lead = (c & 7) == 0;
            if (8 * c < nope) {  // uniform over the block's 8 lanes
                // No clamp to +-448 before the conversion: .satfinite maps
                // every finite value above 448 and +-inf to +-448, keeps NaN,
                // and leaves smaller values alone, as the clamp would.
                float y[8];
                if constexpr (UE8M0) {
                    const float a = fmaxf(am, 1.0e-4f);
                    const int e = ceil_log2_div_const(a, 0x600000u, 8);  // / 448
                    const uint64_t pw2 = splat_f32x2(exp2_int(-e));
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {
                        y[j] = x[j];
                        y[j + 1] = x[j + 1];
                        mul2_rn(y[j], y[j + 1], pw2);
                    }
                    if (lead) scl[c / 8] = (uint8_t)min(max(e + 127, 0), 255);
                } else {
                    const float a = fmaxf(am, 1.0e-12f);
                    const float sc = __fdiv_rn(a, 448.0f);
#pragma unroll
                    for (int j = 0; j < 8; ++j) y[j] = __fdiv_rn(x[j], sc);
                    if (lead) *reinterpret_cast<float*>(scl + 4 * (c / 8)) = sc;
                }
                uint2 q;
                q.x = cvt_e4m3x2(y[0], y[1]) | (cvt_e4m3x2(y[2], y[3]) << 16);
                q.y = cvt_e4m3x2(y[4], y[5]) | (cvt_e4m3x2(y[6], y[7]) << 16);
                st_v2(data + 8 * c, q);
            } else {
                st_v4(data + 16 * c - nope, w);  // rope tail: bf16 verbatim
                if (lead) {  // rope blocks carry a zero scale slot
                    if constexpr (UE8M0) {
                        scl[c / 8] = 0;
                    } else {
                        *reinterpret_cast<uint32_t*>(scl + 4 * (c / 8)) = 0;
                    }
                }
            }
        }
    }
}

// Lanes per token of the MXFP4 insert: two 16-byte chunks per lane where the
// row allows it (halving the per-token slot, address and branch work of one
// chunk per lane), at least the 4 lanes of one 32-element block.  In the insert a
// lane holds adjacent chunks, so a block spans 4 / chunks-per-lane lanes (2 at
// 128 dims: one shuffle step) and the lane's codes leave in one store.
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
    constexpr int LPB = CPL >= 4 ? 1 : 4 / CPL;   // lanes per 32-element block
    constexpr int VB = D / 2;
    static_assert(CPL * LANES == CHUNKS && (CPL == 1 || CPL == 2 || CPL == 4), "chunks per lane");

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
            // the lane's CPL chunks are adjacent: the second 16-byte load of a
            // 32-byte sector hits in L1
            const uint4* row = reinterpret_cast<const uint4*>(k + t * k_row_stride) + CPL * gl;
#pragma unroll
            for (int i = 0; i < CPL; ++i) v[u][i] = __ldg(row + i);
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

        float x[CPL][8];
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const uint4 w = v[u][i];
            const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                x[i][2 * h] = bf16_lo(q[h]);
                x[i][2 * h + 1] = bf16_hi(q[h]);
            }
        }
        // A lane's chunks all lie in one block; fmaxf passes over NaN, as an
        // ordered "a > amax" scan does.
        float am = 0.0f;
#pragma unroll
        for (int i = 0; i < CPL; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) am = fmaxf(am, fabsf(x[i][j]));
#pragma unroll
        for (int m = 1; m < LPB; m <<= 1) am = fmaxf(am, __shfl_xor_sync(gmask, am, m));
        const float a = fmaxf(am, 1.0e-4f);
        const int e = ceil_log2_div_const(a, 0x400000u, 2);  // / 6
        const uint64_t pw2 = splat_f32x2(exp2_int(-e));
        uint32_t words[CPL];
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            uint32_t cd[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float lo = x[i][2 * j], hi = x[i][2 * j + 1];
                mul2_rn(lo, hi, pw2);
                cd[j] = cvt_e2m1x2(lo, hi);
            }
            words[i] = __byte_perm(__byte_perm(cd[0], cd[1], 0x0040),
                                   __byte_perm(cd[2], cd[3], 0x0040), 0x5410);
        }
        uint8_t* vp = vals + 4 * CPL * gl;
        if constexpr (CPL == 1) {
            *reinterpret_cast<uint32_t*>(vp) = words[0];
        } else if constexpr (CPL == 2) {
            *reinterpret_cast<uint2*>(vp) = make_uint2(words[0], words[1]);
        } else {
            *reinterpret_cast<uint4*>(vp) = make_uint4(words[0], words[1], words[2], words[3]);
        }
        // the block's first lane writes its scale byte
        if (gl % LPB == 0) scl[CPL * gl / 4] = (uint8_t)min(max(e + 127, 0), 254);
    }
}

// ---- FP8 indexer record --------------------------------------------------------------
//
// TokenSpeed write_deepseek_v4_indexer_fp8_cache (the "[values | fp32 scale]"
// page layout) with the rule of _fp8_e4m3_pow2_bytes: one power-of-two
// binary32 scale per token, 2^ceil(log2(max(amax / 448, 1e-10))) -- the
// quotient is floored, not amax -- and codes e4m3(x / scale), computed as
// x * 2^-e (the same single rounding of the same exact value).  Lanes as the
// MXFP4 insert; the row amax is a packed bf16x2 max per lane, then a float
// shuffle-max over the token's lanes.
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

        uint32_t mp = absmax_bf16x8_pair(v[u][0]);
#pragma unroll
        for (int i = 1; i < CPL; ++i) mp = bmax2(mp, absmax_bf16x8_pair(v[u][i]));
        float am = absmax_of_pair(mp);
#pragma unroll
        for (int m = 1; m < LANES; m <<= 1) am = fmaxf(am, __shfl_xor_sync(gmask, am, m));
        const float q = fmaxf(__fdiv_rn(am, 448.0f), 1.0e-10f);
        const int e = ceil_log2_pos(q);
        const uint64_t pw2 = splat_f32x2(inv_pow2_scale(e));  // codes e4m3(x / 2^e)
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
// paged store of 128-dim indexer keys.  Four lanes per key, eight keys per
// warp; lane g holds the chunk A = dims [16g, 16g + 16) of the un-rotated half
// and the chunk B = dims [64 + 16g, 64 + 16g + 16) of the RoPE half, so every
// lane rotates eight pairs.  The multiplies run on packed binary32 pairs
// (mul.rn.f32x2: each half the scalar IEEE product), with the pairs chosen so
// that a packed multiply does the same operation on two elements; a sum or
// difference of two products is a scalar add.rn / sub.rn, which the compiler
// never fuses with the products (a packed add after packed products may be
// contracted into a fused multiply-add, which rounds once less).
//  * Emission: slot >= 0 and the token closes its compress group,
//    (pos + 1) % ratio == 0 (TokenSpeed _compress_v4_state_windows_capturable's
//    valid_token rule); other rows are not read (except that with ratio 1,
//    where every row with a slot writes, the row is loaded with the slot).
//  * RMSNorm in binary32, every operation rounded once (no contraction): the
//    sum of squares is a pairwise sum (recursive halving of the index range):
//    each half of the row is a tree over its four 16-dim chunks -- a 4-level
//    tree in the lane (the two halves side by side in one packed pair), then
//    xor-shuffles over 1 and 2 lanes -- and the sum is the two halves' sum.
//    variance = sum * 2^-7 (= sum / 128 exactly); r = 1 / sqrt(variance + eps)
//    as an IEEE binary32 square root then an IEEE reciprocal (= the IEEE
//    quotient 1 / s); y = (x * r) * weight.
//  * GPT-J RoPE (TokenSpeed _apply_gptj_rope_tail_rows) on chunk B at the
//    cos_sin row of the group's first position floor(pos / ratio) * ratio.
//  * MXFP4 record (a 32-block is one chunk of two lanes) or FP8 indexer record
//    (row amax), with the inserts' rules; the scale exponents are read off the
//    binary32 amax without dividing (exact for any normal binary32 amax, as
//    for bf16: see ceil_log2_div_const).
// Keys of a warp that do not write still take part in every shuffle.
constexpr int kKeyLanes = 4;

__device__ __forceinline__ float2 f2_op_mul(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
        "mul.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 f2_op_add(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
        "add.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// One key's state between the stages of the kernel below.
struct NormRopeKey {
    bool act;
    int64_t sl, pos, prow;
    uint4 ka0, ka1, kb0, kb1;  // chunks A and B of the bf16 row
    float4 c0, c1, s0, s1;     // cos and sin of chunk B's eight pairs
};

__device__ __forceinline__ void nrs_load_row(const NormRopeParams& p, int64_t t, int gl,
                                             NormRopeKey& k) {
    const uint16_t* row = p.k + t * p.k_row_stride + 16 * gl;
    k.ka0 = ld_stream_v4(row);
    k.ka1 = ld_stream_v4(row + 8);
    k.kb0 = ld_stream_v4(row + 64);
    k.kb1 = ld_stream_v4(row + 72);
}

// Round trip 1: the slot and the position; with ratio 1 (EVERY_ROW: every row
// with a slot writes) the key row too.
template <bool EVERY_ROW>
__device__ __forceinline__ void nrs_load(const NormRopeParams& p, int64_t t, int gl,
                                         NormRopeKey& k) {
    k.act = t < p.num_tokens;
    k.sl = -1;
    k.pos = k.prow = 0;
    k.ka0 = k.ka1 = k.kb0 = k.kb1 = make_uint4(0u, 0u, 0u, 0u);
    if (k.act) {
        k.sl = __ldg(p.slots + t);
        k.pos = __ldg(p.positions + t);
        if (EVERY_ROW) nrs_load_row(p, t, gl, k);
    }
}

// The emission rule and range checks, then round trip 2: the key row (unless
// already loaded) and chunk B's eight cos and eight sin values.
template <bool EVERY_ROW, bool CS_VEC>
__device__ __forceinline__ void nrs_resolve(const NormRopeParams& p, int64_t t, int gl,
                                            NormRopeKey& k) {
    k.act = k.act && k.sl >= 0;
    if (k.act) {
        const int64_t pos = k.pos;
        const uint32_t ratio = (uint32_t)p.ratio;
        bool boundary;
        if (pos >= 0 && pos < 0xFFFFFFFFll) {
            uint32_t q;
            if (p.ratio_shift >= 0) {  // power-of-two ratio: shift and mask
                q = (uint32_t)pos >> p.ratio_shift;
                boundary = ((uint32_t)pos & (ratio - 1u)) == ratio - 1u;
            } else {
                q = (uint32_t)pos / ratio;
                boundary = (uint32_t)pos - q * ratio == ratio - 1u;
            }
            k.prow = (int64_t)q * ratio;
        } else {
            int64_t rem = (pos + 1) % p.ratio;
            if (rem < 0) rem += p.ratio;
            boundary = rem == 0;
            int64_t grp = pos / p.ratio;
            if (pos % p.ratio != 0 && pos < 0) grp -= 1;
            k.prow = grp * p.ratio;
        }
        k.act = boundary;
        if (k.act && (k.sl >= p.num_pages * (int64_t)p.block_size || k.prow < 0 ||
                      k.prow >= p.max_pos)) {
            if (gl == 0 && p.err_count) atomicAdd(p.err_count, 1);
            k.act = false;
        }
    }
    k.c0 = k.c1 = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
    k.s0 = k.s1 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (k.act) {
        if (!EVERY_ROW) nrs_load_row(p, t, gl, k);
        const float* cs = p.cos_sin + k.prow * p.cs_stride + 8 * gl;
        if (CS_VEC) {
            k.c0 = __ldg(reinterpret_cast<const float4*>(cs));
            k.c1 = __ldg(reinterpret_cast<const float4*>(cs + 4));
            k.s0 = __ldg(reinterpret_cast<const float4*>(cs + 32));
            k.s1 = __ldg(reinterpret_cast<const float4*>(cs + 36));
        } else {
            k.c0 = make_float4(__ldg(cs), __ldg(cs + 1), __ldg(cs + 2), __ldg(cs + 3));
            k.c1 = make_float4(__ldg(cs + 4), __ldg(cs + 5), __ldg(cs + 6), __ldg(cs + 7));
            k.s0 = make_float4(__ldg(cs + 32), __ldg(cs + 33), __ldg(cs + 34), __ldg(cs + 35));
            k.s1 = make_float4(__ldg(cs + 36), __ldg(cs + 37), __ldg(cs + 38), __ldg(cs + 39));
        }
    }
}

// Norm, RoPE, quantize and store one key (every lane of the warp takes part
// in the shuffles).
template <bool FP4>
__device__ __forceinline__ void nrs_compute_store(const NormRopeParams& p, int32_t shift, int gl,
                                                  const NormRopeKey& k) {
    const bool act = k.act;
    // (an inactive key's values are whatever was loaded: its lanes reduce only
    // among themselves and store nothing)
    const uint32_t wa[8] = {k.ka0.x, k.ka0.y, k.ka0.z, k.ka0.w, k.ka1.x, k.ka1.y, k.ka1.z, k.ka1.w};
    const uint32_t wb[8] = {k.kb0.x, k.kb0.y, k.kb0.z, k.kb0.w, k.kb1.x, k.kb1.y, k.kb1.z, k.kb1.w};
    // sum of squares: the pair (A dim i, B dim i) side by side, the 4-level
    // pairwise tree of each chunk in the lane
    float2 t1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 lo = make_float2(bf16_lo(wa[i]), bf16_lo(wb[i]));
        const float2 hi = make_float2(bf16_hi(wa[i]), bf16_hi(wb[i]));
        const float2 sl = f2_op_mul(lo, lo), sh = f2_op_mul(hi, hi);
        t1[i] = make_float2(__fadd_rn(sl.x, sh.x), __fadd_rn(sl.y, sh.y));
    }
    const float2 t2[4] = {f2_op_add(t1[0], t1[1]), f2_op_add(t1[2], t1[3]),
                          f2_op_add(t1[4], t1[5]), f2_op_add(t1[6], t1[7])};
    float2 h = f2_op_add(f2_op_add(t2[0], t2[1]), f2_op_add(t2[2], t2[3]));
    // over the half's four chunks (lanes)
#pragma unroll
    for (int m = 1; m < kKeyLanes; m <<= 1)
        h = f2_op_add(h, make_float2(__shfl_xor_sync(0xFFFFFFFFu, h.x, m),
                                     __shfl_xor_sync(0xFFFFFFFFu, h.y, m)));
    const float variance = __fmul_rn(__fadd_rn(h.x, h.y), 0.0078125f);
    const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(variance, p.eps)));
    const float2 r2 = make_float2(r, r);
    const float4* wv = reinterpret_cast<const float4*>(p.weight) + 4 * gl;
    // chunk A: y = (x r) w, in the pairs (2i, 2i + 1)
    float2 ya[8];
    {
        const float4 w0 = __ldg(wv), w1 = __ldg(wv + 1), w2 = __ldg(wv + 2), w3 = __ldg(wv + 3);
        const float2 w2p[8] = {make_float2(w0.x, w0.y), make_float2(w0.z, w0.w),
                               make_float2(w1.x, w1.y), make_float2(w1.z, w1.w),
                               make_float2(w2.x, w2.y), make_float2(w2.z, w2.w),
                               make_float2(w3.x, w3.y), make_float2(w3.z, w3.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i)
            ya[i] = f2_op_mul(f2_op_mul(make_float2(bf16_lo(wa[i]), bf16_hi(wa[i])), r2), w2p[i]);
    }
    // chunk B: pair j of the lane is (e_j, o_j) = dims (2j, 2j + 1) of the
    // chunk; held as E = (e_2q, e_2q+1) and O = (o_2q, o_2q+1), q = 0..3
    float2 e[4], o[4];
    {
        const float4 w0 = __ldg(wv + 16), w1 = __ldg(wv + 17), w2 = __ldg(wv + 18),
                     w3 = __ldg(wv + 19);
        const float wbv[16] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w,
                               w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
        const float cs[8] = {k.c0.x, k.c0.y, k.c0.z, k.c0.w, k.c1.x, k.c1.y, k.c1.z, k.c1.w};
        const float sn[8] = {k.s0.x, k.s0.y, k.s0.z, k.s0.w, k.s1.x, k.s1.y, k.s1.z, k.s1.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // words 2q, 2q + 1 hold pairs 2q, 2q + 1: (e, o) as (lo, hi)
            const float2 ex = make_float2(bf16_lo(wb[2 * q]), bf16_lo(wb[2 * q + 1]));
            const float2 ox = make_float2(bf16_hi(wb[2 * q]), bf16_hi(wb[2 * q + 1]));
            const float2 ey = f2_op_mul(f2_op_mul(ex, r2),
                                        make_float2(wbv[4 * q], wbv[4 * q + 2]));
            const float2 oy = f2_op_mul(f2_op_mul(ox, r2),
                                        make_float2(wbv[4 * q + 1], wbv[4 * q + 3]));
            const float2 c = make_float2(cs[2 * q], cs[2 * q + 1]);
            const float2 s = make_float2(sn[2 * q], sn[2 * q + 1]);
            const float2 ec = f2_op_mul(ey, c), os = f2_op_mul(oy, s);
            const float2 es = f2_op_mul(ey, s), oc = f2_op_mul(oy, c);
            e[q] = make_float2(__fsub_rn(ec.x, os.x), __fsub_rn(ec.y, os.y));
            o[q] = make_float2(__fadd_rn(es.x, oc.x), __fadd_rn(es.y, oc.y));
        }
    }
    float aa = 0.0f, ab = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) aa = fmaxf(aa, fmaxf(fabsf(ya[i].x), fabsf(ya[i].y)));
#pragma unroll
    for (int q = 0; q < 4; ++q)
        ab = fmaxf(ab, fmaxf(fmaxf(fabsf(e[q].x), fabsf(e[q].y)),
                             fmaxf(fabsf(o[q].x), fabsf(o[q].y))));
    int64_t off = 0;
    uint8_t* base = p.cache;
    if (act) {
        const int64_t page = div_block(k.sl, p.block_size, shift, off);
        base = p.cache + page * p.page_stride;
    }
    // byte / code order of chunk B: dims (2j, 2j + 1) = (e_j, o_j)
    if constexpr (FP4) {
        // 32-blocks: chunk A of lanes 0-1 / 2-3 (blocks 0, 1), chunk B (blocks 2, 3)
        aa = fmaxf(aa, __shfl_xor_sync(0xFFFFFFFFu, aa, 1));
        ab = fmaxf(ab, __shfl_xor_sync(0xFFFFFFFFu, ab, 1));
        const int ea = ceil_log2_div_const(fmaxf(aa, 1.0e-4f), 0x400000u, 2);  // / 6
        const int eb = ceil_log2_div_const(fmaxf(ab, 1.0e-4f), 0x400000u, 2);
        const float2 pa = make_float2(exp2_int(-ea), exp2_int(-ea));
        const float2 pb = make_float2(exp2_int(-eb), exp2_int(-eb));
        uint32_t qa[2] = {0u, 0u}, qb[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 v = f2_op_mul(ya[i], pa);
            qa[i / 4] |= (cvt_e2m1x2(v.x, v.y) & 0xFFu) << (8 * (i % 4));
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 ve = f2_op_mul(e[q], pb), vo = f2_op_mul(o[q], pb);
            // pairs 2q and 2q + 1: bytes 2q, 2q + 1 of the chunk
            const uint32_t b0 = cvt_e2m1x2(ve.x, vo.x) & 0xFFu, b1 = cvt_e2m1x2(ve.y, vo.y) & 0xFFu;
            qb[q / 2] |= (b0 | (b1 << 8)) << (16 * (q % 2));
        }
        if (act) {
            uint8_t* vals = base + off * 64;
            *reinterpret_cast<uint2*>(vals + 8 * gl) = make_uint2(qa[0], qa[1]);
            *reinterpret_cast<uint2*>(vals + 32 + 8 * gl) = make_uint2(qb[0], qb[1]);
            if ((gl & 1) == 0) {
                uint8_t* scl = base + (int64_t)p.block_size * 64 + off * 4 + gl / 2;
                scl[0] = (uint8_t)min(max(ea + 127, 0), 254);
                scl[2] = (uint8_t)min(max(eb + 127, 0), 254);
            }
        }
    } else {
        float a = fmaxf(aa, ab);
#pragma unroll
        for (int m = 1; m < kKeyLanes; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, m));
        // max(a / 448, 1e-10) then ceil(log2): the floor's exponent is -33
        const int ex = max(ceil_log2_div_const(a, 0x600000u, 8), -33);
        const float pwf = inv_pow2_scale(ex);  // codes e4m3(y / 2^e)
        const float2 pw = make_float2(pwf, pwf);
        uint32_t qa[4], qb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 v0 = f2_op_mul(ya[2 * i], pw), v1 = f2_op_mul(ya[2 * i + 1], pw);
            qa[i] = cvt_e4m3x2(v0.x, v0.y) | (cvt_e4m3x2(v1.x, v1.y) << 16);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 ve = f2_op_mul(e[q], pw), vo = f2_op_mul(o[q], pw);
            // dims 4q .. 4q + 3 of the chunk: e_2q, o_2q, e_2q+1, o_2q+1
            qb[q] = cvt_e4m3x2(ve.x, vo.x) | (cvt_e4m3x2(ve.y, vo.y) << 16);
        }
        if (act) {
            uint8_t* vals = base + off * 128;
            *reinterpret_cast<uint4*>(vals + 16 * gl) = make_uint4(qa[0], qa[1], qa[2], qa[3]);
            *reinterpret_cast<uint4*>(vals + 64 + 16 * gl) = make_uint4(qb[0], qb[1], qb[2], qb[3]);
            if (gl == 0)
                *reinterpret_cast<float*>(base + (int64_t)p.block_size * 128 + off * 4) = exp2_int(ex);
        }
    }
}

#ifndef PSK_NORM_ROPE_UNROLL
#define PSK_NORM_ROPE_UNROLL 1
#endif
// Resident CTAs per SM asked of the compiler.  On the 1,048,576-key store
// (one key per group): four (64 registers, 16 bytes spilled) ran 100.4 us,
// no request (78 registers, three CTAs) 104.5 us, one (104 registers) 131 us.
#ifndef PSK_NORM_ROPE_MIN_CTAS
#define PSK_NORM_ROPE_MIN_CTAS 4
#endif
#define PSK_NR_BOUNDS __launch_bounds__(kThreads, PSK_NORM_ROPE_MIN_CTAS)

// U keys per 4-lane group: all of the keys' first-round loads are issued
// before any is used, then all second-round loads, then the arithmetic.
template <bool FP4, bool EVERY_ROW, bool CS_VEC, int U>
__global__ void PSK_NR_BOUNDS norm_rope_store_kernel(NormRopeParams p,
                                                                   int32_t shift) {
    const int gl = (threadIdx.x & 31) % kKeyLanes;
    const int64_t g = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / kKeyLanes;
    const int64_t ngroups = (int64_t)gridDim.x * kThreads / kKeyLanes;
    pdl_wait();
    pdl_launch_dependents();
    NormRopeKey k[U];
#pragma unroll
    for (int u = 0; u < U; ++u) nrs_load<EVERY_ROW>(p, g + u * ngroups, gl, k[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) nrs_resolve<EVERY_ROW, CS_VEC>(p, g + u * ngroups, gl, k[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) nrs_compute_store<FP4>(p, shift, gl, k[u]);
}

// One token per lane group: with the 32-register bound above, a 1M-token
// insert at 512 dims ran 271 us against 275-285 us for two tokens per group
// (40-46 registers) and 277 us for four (64 registers); at the batch sizes of a
// step two tokens per group ran one 2 us event quantum slower on the
// 16384-token prefill (12.3 against 10.2 us), the mixed and the decode batch.
template <int D, bool UE8M0>
cudaError_t fp8_insert_dispatch(const InsertParams& p, cudaStream_t stream) {
    constexpr int UNROLL = 1;
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
    constexpr int U = PSK_NORM_ROPE_UNROLL;
    // kKeyLanes lanes per key, U keys per lane group (keys g, g + G, ... for G groups)
    const int64_t groups = (p.num_tokens + U - 1) / U;
    const int64_t blocks = (groups * kKeyLanes + kThreads - 1) / kThreads;
    const int32_t shift = log2_if_pow2(p.block_size);
    const bool every = p.ratio == 1;
    const bool cs_vec = (reinterpret_cast<uintptr_t>(p.cos_sin) & 15) == 0 && p.cs_stride % 4 == 0;
    using Kern = void (*)(NormRopeParams, int32_t);
    // [fp4][every row][vector cos/sin]
    static const Kern kTable[2][2][2] = {
        {{norm_rope_store_kernel<false, false, false, U>, norm_rope_store_kernel<false, false, true, U>},
         {norm_rope_store_kernel<false, true, false, U>, norm_rope_store_kernel<false, true, true, U>}},
        {{norm_rope_store_kernel<true, false, false, U>, norm_rope_store_kernel<true, false, true, U>},
         {norm_rope_store_kernel<true, true, false, U>, norm_rope_store_kernel<true, true, true, U>}}};
    NormRopeParams q = p;
    q.ratio_shift = log2_if_pow2(p.ratio);
    const Kern kern = kTable[p.record == 1][every][cs_vec];
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), 0, stream, q, shift);
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
