// gather.cu -- index-keyed dequantize-and-gather.
//
// Per-row math: TokenSpeed deepseek_v4_ops.py,
// dequantize_deepseek_v4_fp8_ds_mla_cache (fp8_ds_mla) and
// read_deepseek_v4_indexer_mxfp4_cache (MXFP4); index form of vLLM
// deepseek_v41 ops dequantize_and_gather_k_cache.
//
// Design (HBM-bound: ~584 B read + 1024 B written per fp8 row):
//  * A group of LANES lanes owns one output row (one (token, column) pair);
//    every lane owns 16-byte output chunks (8 bf16), so a 512-dim row is one
//    coalesced 512-byte store instruction per half row, issued as a streaming
//    (evict-first) store so the gathered output does not push reused cache
//    rows out of L2.
//  * The fp8 record is read as 8-byte chunks (nope) and 16-byte chunks (rope)
//    straight from the page; the scale byte of each 64-block is a broadcast
//    load within the block's lanes.
//  * Decode: cvt.rn.f16x2.e4m3x2 (exact), binary32 multiply by the
//    power-of-two scale, cvt.rn.bf16x2.f32.
//  * Each group handles UNROLL rows per step with every load issued first;
//    the grid is a persistent multiple of the SM count and groups stride
//    over the flattened (row, column) space.
//  * Invalid slots (negative or beyond the cache) produce zero rows.
#include "launch.h"
#include "psk_common.cuh"

namespace psk {
namespace {

constexpr int kThreads = 256;

struct RowAddr {
    int64_t t;
    int32_t j;
    int64_t slot;  // -1 = zero row
};

__device__ __forceinline__ RowAddr row_of(const GatherParams& p, int64_t it, int64_t capacity,
                                          bool small) {
    RowAddr a;
    if (small) {
        const uint32_t ui = (uint32_t)it, uc = (uint32_t)p.cols;
        a.t = ui / uc;
        a.j = (int32_t)(ui - (uint32_t)a.t * uc);
    } else {
        a.t = it / p.cols;
        a.j = (int32_t)(it - a.t * p.cols);
    }
    const int32_t s = __ldg(p.idx + a.t * p.idx_stride + a.j);
    a.slot = (s < 0 || (int64_t)s >= capacity) ? -1 : s;
    return a;
}

template <int D, bool UE8M0, int UNROLL>
__global__ void __launch_bounds__(kThreads)
gather_fp8_kernel(GatherParams p) {
    constexpr int CHUNKS = D / 8;
    constexpr int LANES = CHUNKS < kWarp ? CHUNKS : kWarp;
    constexpr int CPL = CHUNKS / LANES;
    constexpr int NBLK = D / 64;
    constexpr int SDIM = UE8M0 ? NBLK : 4 * NBLK;

    const int lane = threadIdx.x & 31;
    const int gl = lane % LANES;
    const int64_t gid = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / LANES;
    const int64_t ngroups = (int64_t)gridDim.x * kThreads / LANES;
    const int64_t items = p.rows * (int64_t)p.cols;
    const int64_t capacity = p.num_pages * (int64_t)p.block_size;
    const bool small = items <= 0xFFFFFFFFll;
    const int nope = D - p.rope_dim;
    const int64_t ts = nope + 2 * p.rope_dim;

    for (int64_t it0 = gid * UNROLL; it0 < items; it0 += ngroups * UNROLL) {
        RowAddr ra[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t it = it0 + u;
            if (it < items) {
                ra[u] = row_of(p, it, capacity, small);
            } else {
                ra[u].t = -1;
                ra[u].slot = -1;
            }
        }
        uint4 raw[UNROLL][CPL];
        float sc[UNROLL][CPL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            if (ra[u].slot < 0) continue;
            const int64_t page = ra[u].slot / p.block_size;
            const int64_t off = ra[u].slot - page * p.block_size;
            const uint8_t* base = p.cache + page * p.page_stride;
            const uint8_t* data = base + off * ts;
            const uint8_t* scl = base + (int64_t)p.block_size * ts + off * SDIM;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int c = gl + i * LANES;
                if (8 * c < nope) {
                    const uint2 w = ld_nc_v2(data + 8 * c);
                    raw[u][i] = make_uint4(w.x, w.y, 0u, 0u);
                    if constexpr (UE8M0) {
                        sc[u][i] = ue8m0_scale(ld_nc_u8(scl + c / 8));
                    } else {
                        sc[u][i] = __uint_as_float(ld_nc_u32(scl + 4 * (c / 8)));
                    }
                } else {
                    raw[u][i] = ld_nc_v4(data + 16 * c - nope);
                    sc[u][i] = 0.0f;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            if (ra[u].t < 0) continue;
            uint16_t* orow = p.out + ra[u].t * p.out_stride_t + (int64_t)ra[u].j * p.out_stride_j;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int c = gl + i * LANES;
                uint4 o;
                if (ra[u].slot < 0) {
                    o = make_uint4(0u, 0u, 0u, 0u);
                } else if (8 * c < nope) {
                    const float s = sc[u][i];
                    const uint32_t h0 = cvt_e4m3x2_to_f16x2(raw[u][i].x & 0xFFFFu);
                    const uint32_t h1 = cvt_e4m3x2_to_f16x2(raw[u][i].x >> 16);
                    const uint32_t h2 = cvt_e4m3x2_to_f16x2(raw[u][i].y & 0xFFFFu);
                    const uint32_t h3 = cvt_e4m3x2_to_f16x2(raw[u][i].y >> 16);
                    o.x = pack_bf16x2(__fmul_rn(f16_lo(h0), s), __fmul_rn(f16_hi(h0), s));
                    o.y = pack_bf16x2(__fmul_rn(f16_lo(h1), s), __fmul_rn(f16_hi(h1), s));
                    o.z = pack_bf16x2(__fmul_rn(f16_lo(h2), s), __fmul_rn(f16_hi(h2), s));
                    o.w = pack_bf16x2(__fmul_rn(f16_lo(h3), s), __fmul_rn(f16_hi(h3), s));
                } else {
                    o = raw[u][i];
                }
                st_stream_v4(orow + 8 * c, o);
            }
        }
    }
}

template <int D, int UNROLL>
__global__ void __launch_bounds__(kThreads)
gather_mxfp4_kernel(GatherParams p) {
    constexpr int CHUNKS = D / 8;
    constexpr int LANES = CHUNKS < kWarp ? CHUNKS : kWarp;
    constexpr int CPL = CHUNKS / LANES;
    constexpr int VB = D / 2, SB = D / 32;

    const int lane = threadIdx.x & 31;
    const int gl = lane % LANES;
    const int64_t gid = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / LANES;
    const int64_t ngroups = (int64_t)gridDim.x * kThreads / LANES;
    const int64_t items = p.rows * (int64_t)p.cols;
    const int64_t capacity = p.num_pages * (int64_t)p.block_size;
    const bool small = items <= 0xFFFFFFFFll;

    for (int64_t it0 = gid * UNROLL; it0 < items; it0 += ngroups * UNROLL) {
        RowAddr ra[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t it = it0 + u;
            if (it < items) {
                ra[u] = row_of(p, it, capacity, small);
            } else {
                ra[u].t = -1;
                ra[u].slot = -1;
            }
        }
        uint32_t raw[UNROLL][CPL];
        float sc[UNROLL][CPL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            if (ra[u].slot < 0) continue;
            const int64_t page = ra[u].slot / p.block_size;
            const int64_t off = ra[u].slot - page * p.block_size;
            const uint8_t* base = p.cache + page * p.page_stride;
            const uint8_t* vals = base + off * VB;
            const uint8_t* scl = base + (int64_t)p.block_size * VB + off * SB;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int c = gl + i * LANES;
                raw[u][i] = ld_nc_u32(vals + 4 * c);
                sc[u][i] = ue8m0_scale(ld_nc_u8(scl + c / 4));
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            if (ra[u].t < 0) continue;
            uint16_t* orow = p.out + ra[u].t * p.out_stride_t + (int64_t)ra[u].j * p.out_stride_j;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int c = gl + i * LANES;
                uint4 o;
                if (ra[u].slot < 0) {
                    o = make_uint4(0u, 0u, 0u, 0u);
                } else {
                    const float s = sc[u][i];
                    const uint32_t w = raw[u][i];
                    uint32_t r[4];
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const uint32_t h = cvt_e2m1x2_to_f16x2((w >> (8 * b)) & 0xFFu);
                        r[b] = pack_bf16x2(__fmul_rn(f16_lo(h), s), __fmul_rn(f16_hi(h), s));
                    }
                    o = make_uint4(r[0], r[1], r[2], r[3]);
                }
                st_stream_v4(orow + 8 * c, o);
            }
        }
    }
}

template <typename K>
int64_t persistent_blocks(K kernel, int64_t groups_needed, int lanes) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t full = (int64_t)sm_count() * per_sm;
    const int64_t need = (groups_needed * lanes + kThreads - 1) / kThreads;
    return need < full ? need : full;
}

template <int D, bool UE8M0>
cudaError_t gather_fp8_dispatch(const GatherParams& p, cudaStream_t stream) {
    constexpr int UNROLL = 2;
    constexpr int LANES = (D / 8) < kWarp ? (D / 8) : kWarp;
    const int64_t items = p.rows * (int64_t)p.cols;
    auto kern = gather_fp8_kernel<D, UE8M0, UNROLL>;
    const int64_t blocks = persistent_blocks(kern, (items + UNROLL - 1) / UNROLL, LANES);
    kern<<<(unsigned)blocks, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t gather_mxfp4_dispatch(const GatherParams& p, cudaStream_t stream) {
    constexpr int UNROLL = 4;
    constexpr int LANES = (D / 8) < kWarp ? (D / 8) : kWarp;
    const int64_t items = p.rows * (int64_t)p.cols;
    auto kern = gather_mxfp4_kernel<D, UNROLL>;
    const int64_t blocks = persistent_blocks(kern, (items + UNROLL - 1) / UNROLL, LANES);
    kern<<<(unsigned)blocks, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream) {
    if (p.record == 0) {
        const bool ue = p.is_ue8m0 != 0;
        switch (p.head_dim) {
            case 64: return ue ? gather_fp8_dispatch<64, true>(p, stream) : gather_fp8_dispatch<64, false>(p, stream);
            case 128: return ue ? gather_fp8_dispatch<128, true>(p, stream) : gather_fp8_dispatch<128, false>(p, stream);
            case 256: return ue ? gather_fp8_dispatch<256, true>(p, stream) : gather_fp8_dispatch<256, false>(p, stream);
            case 512: return ue ? gather_fp8_dispatch<512, true>(p, stream) : gather_fp8_dispatch<512, false>(p, stream);
            case 1024: return ue ? gather_fp8_dispatch<1024, true>(p, stream) : gather_fp8_dispatch<1024, false>(p, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (p.head_dim) {
        case 32: return gather_mxfp4_dispatch<32>(p, stream);
        case 64: return gather_mxfp4_dispatch<64>(p, stream);
        case 128: return gather_mxfp4_dispatch<128>(p, stream);
        case 256: return gather_mxfp4_dispatch<256>(p, stream);
        case 512: return gather_mxfp4_dispatch<512>(p, stream);
        case 1024: return gather_mxfp4_dispatch<1024>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace psk
