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

}  // namespace

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
