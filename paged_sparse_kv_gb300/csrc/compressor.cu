// compressor.cu -- the compressed-KV producer: the compressor's residual state
// and the window-pooled, normalised, rotated and quantised compressed rows.
//
// TokenSpeed deepseek_v4_ops.py: save_deepseek_v4_compressor_state, and
// deepseek_v4_csa_compress_kv_cache_insert (ratio 4, an overlapping 8-wide
// window) / deepseek_v4_hca_compress_kv_cache_insert (ratio 128), whose torch
// form is _compress_v4_state_windows_capturable followed by
// _write_fp8_ds_mla_cache_rows_capturable.
//
// Every floating-point step is the IEEE binary32 operation the CPU oracle
// performs, in the same order, without contraction: the window softmax (max,
// then the exps summed in window order, then each weight = exp / sum and the
// weighted kv summed in window order), the RMSNorm (pairwise sum of squares,
// IEEE square root and reciprocal) and GPT-J RoPE.  exp itself is
// cw_exp below -- Cody and Waite's argument reduction and the Taylor series --
// the same operation sequence as the oracle's, not a library call, so the two
// agree to the bit.
#include "compressor.h"
#include "psk_common.cuh"

namespace psk {
namespace {

constexpr int kThreads = 256;  // state writer

// exp of a binary32 by Cody and Waite's argument reduction and the Taylor
// series to r^7/7!, evaluated by Horner with fused multiply-adds: k = nearest
// integer to x / ln 2, r = x - k * ln2_hi - k * ln2_lo (ln2_hi with 16
// significant bits), result = p(r) * 2^k with one rounding.
__device__ __forceinline__ float cw_exp(float x) {
    if (x != x) return x;
    if (x > 88.7228f) return __int_as_float(0x7F800000);
    if (x < -103.98f) return 0.0f;
    const float k = rintf(__fmul_rn(x, 1.44269504f));
    float r = __fmaf_rn(-k, 0.693145751953125f, x);
    r = __fmaf_rn(-k, 1.42860677e-06f, r);
    float p = 1.98412698e-04f;
    p = __fmaf_rn(p, r, 1.38888889e-03f);
    p = __fmaf_rn(p, r, 8.33333333e-03f);
    p = __fmaf_rn(p, r, 4.16666667e-02f);
    p = __fmaf_rn(p, r, 1.66666667e-01f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int ki = (int)k;
    if (ki < -126) return __fmul_rn(__fmul_rn(p, exp2_int(ki + 64)), exp2_int(-64));
    if (ki > 127) return __fmul_rn(__fmul_rn(p, exp2_int(ki - 1)), 2.0f);
    return __fmul_rn(p, exp2_int(ki));
}

// ---- compressor state ----------------------------------------------------------------
//
// state[slot] = [kv[t], score[t] + ape[pos % ratio]] (binary32 adds), one warp
// per token, 16-byte loads and stores.
__global__ void __launch_bounds__(kThreads) save_state_kernel(SaveStateParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t t = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / kWarp;
    pdl_wait();
    pdl_launch_dependents();
    if (t >= p.num_tokens) return;
    const int64_t s = __ldg(p.slots + t);
    if (s < 0) return;
    if (s >= p.num_pages * (int64_t)p.block_size) {
        if (lane == 0 && p.err_count) atomicAdd(p.err_count, 1);
        return;
    }
    int64_t a = __ldg(p.positions + t) % p.ratio;
    if (a < 0) a += p.ratio;
    const float4* kv = reinterpret_cast<const float4*>(p.kv + t * p.in_stride);
    const float4* sc = reinterpret_cast<const float4*>(p.score + t * p.in_stride);
    const float4* ap = reinterpret_cast<const float4*>(p.ape + a * p.state_width);
    float4* row = reinterpret_cast<float4*>(p.state + s * 2 * (int64_t)p.state_width);
    const int n4 = p.state_width / 4;
    for (int i = lane; i < n4; i += kWarp) {
        const float4 k4 = __ldg(kv + i), s4 = __ldg(sc + i), a4 = __ldg(ap + i);
        row[i] = k4;
        row[n4 + i] = make_float4(__fadd_rn(s4.x, a4.x), __fadd_rn(s4.y, a4.y),
                                  __fadd_rn(s4.z, a4.z), __fadd_rn(s4.w, a4.w));
    }
}

// ---- compressed rows ------------------------------------------------------------------
//
// One CTA per token.  THREADS = 128 (four columns per thread; windows of at
// most 8 rows are loaded into registers in one round trip) or 512 (one column
// per thread, the window streamed with loads issued eight rows ahead) -- the
// latter for long windows, which have few tokens to spread over the GPU.
// Every column's softmax is computed by one thread in window order, so the
// split of columns does not change any result.  The normalised row goes
// through shared memory to a common epilogue: 128 threads, four dims each
// (RoPE on the tail, bf16, the fp8_ds_mla record).
constexpr int kMaxWindow = 256;
constexpr int kHead = 512;
constexpr int kRope = 64;
constexpr int kNope = kHead - kRope;

// Score / kv float4 (or float) of column group `col` of window row j.
template <int CPT>
__device__ __forceinline__ void load_slice(const CompressParams& p, int64_t row, int j, int col,
                                           float (&s)[CPT], float (&k)[CPT], bool want_kv) {
    const int off = (p.overlap && j >= p.ratio) ? kHead : 0;
    if (row < 0) {
#pragma unroll
        for (int e = 0; e < CPT; ++e) {
            s[e] = -1.0e30f;
            k[e] = 0.0f;
        }
        return;
    }
    const float* rp = p.state + row * 2 * (int64_t)p.state_width + off + col;
    if constexpr (CPT == 4) {
        const float4 s4 = __ldg(reinterpret_cast<const float4*>(rp + p.state_width));
        s[0] = s4.x; s[1] = s4.y; s[2] = s4.z; s[3] = s4.w;
        if (want_kv) {
            const float4 k4 = __ldg(reinterpret_cast<const float4*>(rp));
            k[0] = k4.x; k[1] = k4.y; k[2] = k4.z; k[3] = k4.w;
        }
    } else {
        s[0] = __ldg(rp + p.state_width);
        if (want_kv) k[0] = __ldg(rp);
    }
}

// One token's compressed row (the whole CTA; every thread calls it).
template <int THREADS, bool REGS>
__device__ __forceinline__ void compress_token(const CompressParams& p, int32_t kv_shift, int64_t t,
                                               int64_t* s_row, float* s_part, float* s_y) {
    constexpr int CPT = kHead / THREADS;  // columns per thread
    constexpr int NW = THREADS / kWarp;
    constexpr int WREG = 8;               // window rows held in registers (REGS)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t ks = __ldg(p.kv_slots + t);
    const int64_t pos = __ldg(p.positions + t);
    int64_t grp = pos / p.ratio;
    if (pos % p.ratio != 0 && pos < 0) grp -= 1;
    const int64_t prow = grp * p.ratio;
    const int32_t r = __ldg(p.t2r + t);
    const int window = (p.overlap ? 2 : 1) * p.ratio;
    const int64_t state_cap = p.state_pages * (int64_t)p.state_bs;
    const int64_t base = p.base ? __ldg(p.base + r) : 0;
    for (int j = tid; j < window; j += THREADS) {
        const int64_t ps = pos - window + 1 + j;
        int64_t row = -1;
        if (ps >= 0) {
            const int64_t lp = ps / p.state_bs - base;
            if (lp >= 0 && lp < p.bt_width) {
                const int32_t entry = __ldg(p.bt + (int64_t)r * p.bt_stride + lp);
                if (entry >= 0) {
                    const int64_t sr = (int64_t)entry * p.state_bs + ps % p.state_bs;
                    if (sr < state_cap) row = sr;
                }
            }
        }
        s_row[j] = row;
    }
    __syncthreads();

    const int col = CPT * tid;
    float mx[CPT], sum[CPT], acc[CPT];
#pragma unroll
    for (int e = 0; e < CPT; ++e) {
        sum[e] = 0.0f;
        acc[e] = 0.0f;
    }
    if (REGS) {
        // the whole window (<= 8 rows) in registers: one round of loads
        float sv[WREG][CPT], kv[WREG][CPT];
#pragma unroll
        for (int j = 0; j < WREG; ++j)
            if (j < window) load_slice<CPT>(p, s_row[j], j, col, sv[j], kv[j], true);
#pragma unroll
        for (int e = 0; e < CPT; ++e) mx[e] = sv[0][e];
#pragma unroll
        for (int j = 1; j < WREG; ++j)
            if (j < window)
#pragma unroll
                for (int e = 0; e < CPT; ++e) mx[e] = sv[j][e] > mx[e] ? sv[j][e] : mx[e];
        float ex[WREG][CPT];
#pragma unroll
        for (int j = 0; j < WREG; ++j)
            if (j < window)
#pragma unroll
                for (int e = 0; e < CPT; ++e) {
                    ex[j][e] = cw_exp(__fsub_rn(sv[j][e], mx[e]));
                    sum[e] = __fadd_rn(sum[e], ex[j][e]);
                }
#pragma unroll
        for (int j = 0; j < WREG; ++j)
            if (j < window)
#pragma unroll
                for (int e = 0; e < CPT; ++e)
                    acc[e] = __fadd_rn(acc[e], __fmul_rn(kv[j][e], __fdiv_rn(ex[j][e], sum[e])));
    } else {
        // streamed: three passes, U rows' loads issued before their use
        constexpr int U = 8;
        for (int j0 = 0; j0 < window; j0 += U) {
            float sv[U][CPT], kd[U][CPT];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (j0 + u < window) load_slice<CPT>(p, s_row[j0 + u], j0 + u, col, sv[u], kd[u], false);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (j0 + u < window)
#pragma unroll
                    for (int e = 0; e < CPT; ++e)
                        mx[e] = (j0 + u == 0) ? sv[u][e] : (sv[u][e] > mx[e] ? sv[u][e] : mx[e]);
        }
        for (int j0 = 0; j0 < window; j0 += U) {
            float sv[U][CPT], kd[U][CPT];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (j0 + u < window) load_slice<CPT>(p, s_row[j0 + u], j0 + u, col, sv[u], kd[u], false);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (j0 + u < window)
#pragma unroll
                    for (int e = 0; e < CPT; ++e)
                        sum[e] = __fadd_rn(sum[e], cw_exp(__fsub_rn(sv[u][e], mx[e])));
        }
        for (int j0 = 0; j0 < window; j0 += U) {
            float sv[U][CPT], kd[U][CPT];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (j0 + u < window) load_slice<CPT>(p, s_row[j0 + u], j0 + u, col, sv[u], kd[u], true);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (j0 + u < window)
#pragma unroll
                    for (int e = 0; e < CPT; ++e) {
                        const float w = __fdiv_rn(cw_exp(__fsub_rn(sv[u][e], mx[e])), sum[e]);
                        acc[e] = __fadd_rn(acc[e], __fmul_rn(kd[u][e], w));
                    }
        }
    }

    // RMSNorm: pairwise sum of squares over the 512 columns -- in the thread
    // (CPT = 4: (a + b) + (c + d)), across the warp's lanes, then a pairwise
    // tree over the warps' partial sums
    float ssq;
    if constexpr (CPT == 4)
        ssq = __fadd_rn(__fadd_rn(__fmul_rn(acc[0], acc[0]), __fmul_rn(acc[1], acc[1])),
                        __fadd_rn(__fmul_rn(acc[2], acc[2]), __fmul_rn(acc[3], acc[3])));
    else
        ssq = __fmul_rn(acc[0], acc[0]);
#pragma unroll
    for (int m = 1; m < kWarp; m <<= 1) ssq = __fadd_rn(ssq, __shfl_xor_sync(0xFFFFFFFFu, ssq, m));
    if (lane == 0) s_part[warp] = ssq;
    __syncthreads();
    float part[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) part[i] = s_part[i];
#pragma unroll
    for (int n = NW / 2; n >= 1; n >>= 1)
#pragma unroll
        for (int i = 0; i < n; ++i) part[i] = __fadd_rn(part[2 * i], part[2 * i + 1]);
    const float variance = __fmul_rn(part[0], 1.0f / kHead);  // exact: a power of two
    const float rr = __frcp_rn(__fsqrt_rn(__fadd_rn(variance, p.eps)));
#pragma unroll
    for (int e = 0; e < CPT; ++e)
        s_y[col + e] = __fmul_rn(__fmul_rn(acc[e], rr), __ldg(p.weight + col + e));
    __syncthreads();
    if (tid < kHead / 4) {  // epilogue: 128 threads (warps 0-3), dims 4i..4i+3
    const int d0 = 4 * tid;
    float y[4] = {s_y[d0], s_y[d0 + 1], s_y[d0 + 2], s_y[d0 + 3]};
    if (d0 >= kNope) {  // GPT-J RoPE at the group's first position
        const float* cs = p.cos_sin + prow * p.cs_stride;
        const int i0 = (d0 - kNope) / 2;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float c = __ldg(cs + i0 + h), sn = __ldg(cs + kRope / 2 + i0 + h);
            const float e = y[2 * h], o = y[2 * h + 1];
            y[2 * h] = __fsub_rn(__fmul_rn(e, c), __fmul_rn(o, sn));
            y[2 * h + 1] = __fadd_rn(__fmul_rn(e, sn), __fmul_rn(o, c));
        }
    }
    // the bf16 row, then the fp8_ds_mla record (64-wide blocks = 16 threads)
    const uint32_t b01 = pack_bf16x2(y[0], y[1]), b23 = pack_bf16x2(y[2], y[3]);
    int64_t off;
    const int64_t page = div_block(ks, p.kv_bs, kv_shift, off);
    constexpr int kTS = kNope + 2 * kRope;  // 576 data bytes per token
    uint8_t* pbase = p.kv_cache + page * p.kv_page_stride;
    uint8_t* data = pbase + off * kTS;
    uint8_t* scl = pbase + (int64_t)p.kv_bs * kTS + off * (kHead / 64);
    uint32_t amb = max(max(b01 & 0x7FFFu, (b01 >> 16) & 0x7FFFu),
                       max(b23 & 0x7FFFu, (b23 >> 16) & 0x7FFFu));
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) amb = max(amb, __shfl_xor_sync(0xFFFFFFFFu, amb, m));
    if (d0 < kNope) {
        const float a = fmaxf(__uint_as_float(amb << 16), 1.0e-4f);
        const int e = ceil_log2_div_const(a, 0x600000u, 8);  // / 448
        const float pw = exp2_int(-e);
        const uint32_t q = cvt_e4m3x2(__fmul_rn(bf16_lo(b01), pw), __fmul_rn(bf16_hi(b01), pw)) |
                           (cvt_e4m3x2(__fmul_rn(bf16_lo(b23), pw), __fmul_rn(bf16_hi(b23), pw))
                            << 16);
        *reinterpret_cast<uint32_t*>(data + d0) = q;
        if ((tid & 15) == 0) scl[tid / 16] = (uint8_t)min(max(e + 127, 0), 255);
    } else {
        *reinterpret_cast<uint2*>(data + kNope + 2 * (d0 - kNope)) = make_uint2(b01, b23);
        if (tid == kNope / 4) scl[kNope / 64] = 0;  // the unused scale slot
    }
    }
}

// Persistent CTAs: each scans contiguous 32-token chunks (warp 0: one
// coalesced read of the chunk's slots and positions, a ballot of the tokens
// that write, counted skips), lists the writing tokens in ascending order in
// shared memory, and processes them one at a time with the whole CTA -- most
// tokens of a batch do not close a group, so no CTA is spent on them.
template <int THREADS, bool REGS>
__global__ void __launch_bounds__(THREADS) compress_kernel(CompressParams p, int32_t kv_shift) {
    __shared__ int64_t s_row[kMaxWindow];
    __shared__ float s_part[THREADS / kWarp];
    __shared__ __align__(16) float s_y[kHead];
    __shared__ int64_t s_list[kWarp];
    __shared__ int s_count;
    const int tid = threadIdx.x, lane = tid & 31;
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t c0 = (int64_t)blockIdx.x * kWarp; c0 < p.num_tokens;
         c0 += (int64_t)gridDim.x * kWarp) {
        if (tid < kWarp) {
            const int64_t t = c0 + lane;
            bool emit = false;
            if (t < p.num_tokens) {
                const int64_t ss = __ldg(p.state_slots + t), ks = __ldg(p.kv_slots + t);
                const int64_t pos = __ldg(p.positions + t);
                if (ss >= 0 && ks >= 0) {
                    int64_t rem = (pos + 1) % p.ratio;
                    if (rem < 0) rem += p.ratio;
                    if (rem == 0) {
                        int64_t grp = pos / p.ratio;
                        if (pos % p.ratio != 0 && pos < 0) grp -= 1;
                        const int64_t prow = grp * p.ratio;
                        const int32_t r = __ldg(p.t2r + t);
                        if (ks >= p.kv_pages * (int64_t)p.kv_bs || prow < 0 || prow >= p.max_pos ||
                            r < 0 || r >= p.num_reqs) {
                            if (p.err_count) atomicAdd(p.err_count, 1);
                        } else {
                            emit = true;
                        }
                    }
                }
            }
            const unsigned mask = __ballot_sync(0xFFFFFFFFu, emit);
            if (emit) s_list[__popc(mask & ((1u << lane) - 1u))] = t;
            if (lane == 0) s_count = __popc(mask);
        }
        __syncthreads();
        const int n = s_count;
        for (int i = 0; i < n; ++i) {
            compress_token<THREADS, REGS>(p, kv_shift, s_list[i], s_row, s_part, s_y);
            __syncthreads();
        }
        __syncthreads();  // every thread has read s_count / s_list before the next scan
    }
}

}  // namespace

cudaError_t launch_save_compressor_state(const SaveStateParams& p, cudaStream_t stream) {
    const int64_t blocks = (p.num_tokens * kWarp + kThreads - 1) / kThreads;
    return launch_pdl(save_state_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, p);
}

cudaError_t launch_compress_kv_insert(const CompressParams& p, cudaStream_t stream) {
    const int window = (p.overlap ? 2 : 1) * p.ratio;
    const int32_t shift = log2_if_pow2(p.kv_bs);
    const int64_t chunks = (p.num_tokens + kWarp - 1) / kWarp;
    auto grid_for = [&](auto kern, int threads) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) !=
                cudaSuccess || per_sm < 1)
            per_sm = 1;
        const int64_t full = (int64_t)sm_count() * per_sm;
        return dim3((unsigned)(chunks < full ? chunks : full));
    };
    if (window <= 8) {
        auto kern = compress_kernel<128, true>;
        return launch_pdl(kern, grid_for(kern, 128), dim3(128), 0, stream, p, shift);
    }
    auto kern = compress_kernel<512, false>;
    return launch_pdl(kern, grid_for(kern, 512), dim3(512), 0, stream, p, shift);
}

}  // namespace psk
