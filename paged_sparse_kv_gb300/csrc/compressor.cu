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
// cw_exp_nonpos below -- Cody and Waite's argument reduction and the Taylor
// series -- the same operation sequence as the oracle's, not a library call,
// so the two agree to the bit.
#include "compressor.h"
#include "psk_common.cuh"

namespace psk {
namespace {

constexpr int kThreads = 256;  // state writer

// exp of a binary32 by Cody and Waite's argument reduction and the Taylor
// series to r^7/7!, evaluated by Horner with fused multiply-adds: k = nearest
// integer to x / ln 2, r = x - k * ln2_hi - k * ln2_lo (ln2_hi with 16
// significant bits), result = p(r) * 2^k with one rounding (two multiplies,
// the second exact or the final one, when 2^k is not a normal binary32).
// Only for x <= 0 or NaN: every argument here is a score minus the window's
// maximum, so the overflow side (x > 88.7228, 2^k above the binary32 range)
// cannot occur and is left out; on this domain the result is the general
// case-by-case function's.  Branch-free, so that a thread's independent exps
// interleave: the core runs on max(x, -103.98) -- x itself inside the range --
// and NaN and underflow are selected at the end.
__device__ __forceinline__ float cw_exp_nonpos(float x) {
    const float xc = fmaxf(x, -103.98f);
    const float k = rintf(__fmul_rn(xc, 1.44269504f));
    float r = __fmaf_rn(-k, 0.693145751953125f, xc);
    r = __fmaf_rn(-k, 1.42860677e-06f, r);
    float p = 1.98412698e-04f;
    p = __fmaf_rn(p, r, 1.38888889e-03f);
    p = __fmaf_rn(p, r, 8.33333333e-03f);
    p = __fmaf_rn(p, r, 4.16666667e-02f);
    p = __fmaf_rn(p, r, 1.66666667e-01f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int ki = (int)k;  // in [-150, 0]
    const bool sub = ki < -126;
    const int a = sub ? ki + 64 : ki;  // in [-126, 0]
    const float f = sub ? __uint_as_float(0x1F800000u) /* 2^-64 */ : 1.0f;
    const float v = __fmul_rn(__fmul_rn(p, __uint_as_float((uint32_t)(a + 127) << 23)), f);
    return x != x ? x : (x < -103.98f ? 0.0f : v);
}

// Packed binary32 pairs (each lane the scalar IEEE operation, round to
// nearest even).  Used only where the product feeds a conversion, a multiply
// or an explicit fma: a packed product feeding a packed add may be contracted
// into a fused multiply-add by the compiler.
__device__ __forceinline__ float2 pk_mul(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 x, y, z;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 y, {%4, %5};\n\t"
        "mul.rn.f32x2 z, x, y;\n\t"
        "mov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float2 pk_fma(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{\n\t.reg .b64 x, y, z, w;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 y, {%4, %5};\n\t"
        "mov.b64 z, {%6, %7};\n\t"
        "fma.rn.f32x2 w, x, y, z;\n\t"
        "mov.b64 {%0, %1}, w;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

__device__ __forceinline__ float2 pk_splat(float v) { return make_float2(v, v); }

// cw_exp_nonpos of two arguments at once: the same operations lane by lane,
// the multiplies and fused multiply-adds issued as packed pairs.
__device__ __forceinline__ void cw_exp2_nonpos(float x0, float x1, float& y0, float& y1) {
    const float2 xc = make_float2(fmaxf(x0, -103.98f), fmaxf(x1, -103.98f));
    const float2 t = pk_mul(xc, pk_splat(1.44269504f));
    const float k0 = rintf(t.x), k1 = rintf(t.y);
    const float2 nk = make_float2(-k0, -k1);
    float2 r = pk_fma(nk, pk_splat(0.693145751953125f), xc);
    r = pk_fma(nk, pk_splat(1.42860677e-06f), r);
    float2 p = pk_splat(1.98412698e-04f);
    p = pk_fma(p, r, pk_splat(1.38888889e-03f));
    p = pk_fma(p, r, pk_splat(8.33333333e-03f));
    p = pk_fma(p, r, pk_splat(4.16666667e-02f));
    p = pk_fma(p, r, pk_splat(1.66666667e-01f));
    p = pk_fma(p, r, pk_splat(0.5f));
    p = pk_fma(p, r, pk_splat(1.0f));
    p = pk_fma(p, r, pk_splat(1.0f));
    const int i0 = (int)k0, i1 = (int)k1;
    const bool s0 = i0 < -126, s1 = i1 < -126;
    const int a0 = s0 ? i0 + 64 : i0, a1 = s1 ? i1 + 64 : i1;
    const float f0 = s0 ? __uint_as_float(0x1F800000u) : 1.0f;
    const float f1 = s1 ? __uint_as_float(0x1F800000u) : 1.0f;
    const float2 v = pk_mul(pk_mul(p, make_float2(__uint_as_float((uint32_t)(a0 + 127) << 23),
                                                  __uint_as_float((uint32_t)(a1 + 127) << 23))),
                            make_float2(f0, f1));
    y0 = x0 != x0 ? x0 : (x0 < -103.98f ? 0.0f : v.x);
    y1 = x1 != x1 ? x1 : (x1 < -103.98f ? 0.0f : v.y);
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
// Windows of at most 8 rows (CSA: ratio 4, overlapping): one CTA of 128
// threads per 32-token chunk, four columns per thread.  After the chunk's scan
// every writing token's window rows are resolved in one round of table
// look-ups; each token's window then reaches the threads through a per-thread
// shared-memory buffer filled by cp.async, so the next token's copies are in
// flight while the current token computes: its scores as soon as the current
// scores have been read, its kv as soon as the current kv have.  Every
// column's softmax is computed by one thread in window order, so neither the
// split of columns nor the pipelining changes any result.  The normalised row
// goes through shared memory to the epilogue: 128 threads, four dims each
// (RoPE on the tail, bf16, the fp8_ds_mla record).  Longer windows take the
// cluster kernel further below.
constexpr int kMaxWindow = 256;
constexpr int kHead = 512;
constexpr int kRope = 64;
constexpr int kNope = kHead - kRope;
constexpr int kWinRows = 8;  // rows of a short window

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's committed copy groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// State row of window row j of a writing token (request r, position pos; the
// request's block-table base offset `base`), or -1: a negative position, a
// logical page outside the table row, a missing page or a row beyond the
// state cache.
__device__ __forceinline__ int64_t window_row(const CompressParams& p, int64_t pos, int32_t r,
                                              int64_t base, int window, int j) {
    const int64_t ps = pos - window + 1 + j;
    if (ps < 0) return -1;
    const int64_t lp = ps / p.state_bs - base;
    if (lp < 0 || lp >= p.bt_width) return -1;
    const int32_t entry = __ldg(p.bt + (int64_t)r * p.bt_stride + lp);
    if (entry < 0) return -1;
    const int64_t sr = (int64_t)entry * p.state_bs + ps % p.state_bs;
    return sr < p.state_pages * (int64_t)p.state_bs ? sr : -1;
}

// Issues this thread's copies of one half of a token's window (its four
// columns of every present row: the scores, or the kv) into its own buffer
// slots: buf[(2 j + half) * THREADS + tid].  The slots hold the previous
// token's values of this thread; `after` is a value computed from all of them,
// and the copies' addresses are made to depend on it, so the copies are issued
// (in program order, hence after those values were read) only once it exists.
template <int THREADS>
__device__ __forceinline__ void prefetch_window(const CompressParams& p, const int64_t* rows,
                                                int window, int half, float4* buf, float after) {
    const int tid = threadIdx.x;
    const float* state = p.state;
    asm volatile("" : "+l"(state) : "f"(after));
#pragma unroll
    for (int j = 0; j < kWinRows; ++j) {
        if (j >= window || rows[j] < 0) continue;
        const int off = (p.overlap && j >= p.ratio) ? kHead : 0;
        const float* rp = state + rows[j] * 2 * (int64_t)p.state_width + off + 4 * tid +
                          (half == 0 ? p.state_width : 0);
        cp_async16(buf + (2 * j + half) * THREADS + tid, rp);
    }
}

// The RMSNorm, RoPE and record of one pooled row (acc: this thread's four
// columns); every thread of the CTA calls it.
template <int THREADS>
__device__ __forceinline__ void finish_token(const CompressParams& p, int32_t kv_shift, int64_t ks,
                                             int64_t prow, const float (&acc)[4], float* s_part,
                                             float* s_y) {
    constexpr int CPT = 4;
    constexpr int NW = THREADS / kWarp;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int col = CPT * tid;
    // RMSNorm: pairwise sum of squares over the 512 columns -- in the thread
    // ((a + b) + (c + d)), across the warp's lanes, then a pairwise tree over
    // the warps' partial sums
    float ssq = __fadd_rn(__fadd_rn(__fmul_rn(acc[0], acc[0]), __fmul_rn(acc[1], acc[1])),
                          __fadd_rn(__fmul_rn(acc[2], acc[2]), __fmul_rn(acc[3], acc[3])));
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

// Persistent CTAs: each scans contiguous CHUNK-token chunks (warp 0: one
// coalesced read of the chunk's slots and positions, a ballot of the tokens
// that write, counted skips), lists the writing tokens in ascending order in
// shared memory with their requests, positions and record slots, resolves
// every listed token's window rows, and pools the tokens one at a time with
// the whole CTA -- most tokens of a batch do not close a group, so no CTA is
// spent on them.
template <int THREADS, int CHUNK>
__global__ void __launch_bounds__(THREADS, 4) compress_kernel(CompressParams p, int32_t kv_shift) {
    static_assert(THREADS * 4 == kHead, "four columns per thread");
    constexpr int CPT = 4;
    __shared__ __align__(16) float4 s_win[2 * kWinRows * THREADS];  // [row][scores | kv][thread]
    __shared__ int64_t s_rows[CHUNK][kWinRows];
    __shared__ int64_t s_tok[CHUNK], s_pos[CHUNK], s_ks[CHUNK], s_prow[CHUNK];
    __shared__ int32_t s_req[CHUNK];
    __shared__ float s_part[THREADS / kWarp];
    __shared__ __align__(16) float s_y[kHead];
    __shared__ int s_count;
    const int tid = threadIdx.x, lane = tid & 31;
    const int window = (p.overlap ? 2 : 1) * p.ratio;
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t c0 = (int64_t)blockIdx.x * CHUNK; c0 < p.num_tokens;
         c0 += (int64_t)gridDim.x * CHUNK) {
        if (tid < kWarp) {
            const int64_t t = c0 + lane;
            bool emit = false;
            int64_t pos = 0, ks = 0, prow = 0;
            int32_t r = 0;
            if (lane < CHUNK && t < p.num_tokens) {
                const int64_t ss = __ldg(p.state_slots + t);
                ks = __ldg(p.kv_slots + t);
                pos = __ldg(p.positions + t);
                if (ss >= 0 && ks >= 0) {
                    int64_t rem = (pos + 1) % p.ratio;
                    if (rem < 0) rem += p.ratio;
                    if (rem == 0) {
                        int64_t grp = pos / p.ratio;
                        if (pos % p.ratio != 0 && pos < 0) grp -= 1;
                        prow = grp * p.ratio;
                        r = __ldg(p.t2r + t);
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
            if (emit) {
                const int k = __popc(mask & ((1u << lane) - 1u));
                s_tok[k] = t;
                s_pos[k] = pos;
                s_ks[k] = ks;
                s_prow[k] = prow;
                s_req[k] = r;
            }
            if (lane == 0) s_count = __popc(mask);
        }
        __syncthreads();
        const int n = s_count;
        // every listed token's window rows: one round of table look-ups
        for (int k = tid; k < n * window; k += THREADS) {
            const int i = k / window, j = k - i * window;
            const int64_t base = p.base ? __ldg(p.base + s_req[i]) : 0;
            s_rows[i][j] = window_row(p, s_pos[i], s_req[i], base, window, j);
        }
        __syncthreads();
        if (n > 0) {
            prefetch_window<THREADS>(p, s_rows[0], window, 0, s_win, 0.0f);
            cp_async_commit();
            prefetch_window<THREADS>(p, s_rows[0], window, 1, s_win, 0.0f);
            cp_async_commit();
        }
        for (int i = 0; i < n; ++i) {
            const bool more = i + 1 < n;
            float mx[CPT], sum[CPT], acc[CPT];
#pragma unroll
            for (int e = 0; e < CPT; ++e) {
                sum[e] = 0.0f;
                acc[e] = 0.0f;
            }
            float ex[kWinRows][CPT];
            {
                // scores: the token's score copies have landed (its kv copies may not)
                cp_async_wait<1>();
                float sv[kWinRows][CPT];
#pragma unroll
                for (int j = 0; j < kWinRows; ++j) {
                    if (j >= window) continue;
                    if (s_rows[i][j] < 0) {
#pragma unroll
                        for (int e = 0; e < CPT; ++e) sv[j][e] = -1.0e30f;
                    } else {
                        const float4 v = s_win[(2 * j) * THREADS + tid];
                        sv[j][0] = v.x; sv[j][1] = v.y; sv[j][2] = v.z; sv[j][3] = v.w;
                    }
                }
#pragma unroll
                for (int e = 0; e < CPT; ++e) mx[e] = sv[0][e];
#pragma unroll
                for (int j = 1; j < kWinRows; ++j)
                    if (j < window)
#pragma unroll
                        for (int e = 0; e < CPT; ++e) mx[e] = sv[j][e] > mx[e] ? sv[j][e] : mx[e];
#pragma unroll
                for (int j = 0; j < kWinRows; ++j)
                    if (j < window) {
#pragma unroll
                        for (int e = 0; e < CPT; e += 2)
                            cw_exp2_nonpos(__fsub_rn(sv[j][e], mx[e]),
                                           __fsub_rn(sv[j][e + 1], mx[e + 1]), ex[j][e],
                                           ex[j][e + 1]);
#pragma unroll
                        for (int e = 0; e < CPT; ++e) sum[e] = __fadd_rn(sum[e], ex[j][e]);
                    }
            }
            // the scores have been read (the exps depend on them): the next
            // token's scores may overwrite them
            if (more)
                prefetch_window<THREADS>(p, s_rows[i + 1], window, 0, s_win,
                                         __fadd_rn(__fadd_rn(sum[0], sum[1]), __fadd_rn(sum[2], sum[3])));
            cp_async_commit();
            // kv: every group but the one just committed has landed
            cp_async_wait<1>();
            {
                // each row's kv read where it is used (fewer live registers)
#pragma unroll
                for (int j = 0; j < kWinRows; ++j) {
                    if (j >= window) continue;
                    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    if (s_rows[i][j] >= 0) v = s_win[(2 * j + 1) * THREADS + tid];
                    const float kv4[CPT] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < CPT; ++e)
                        acc[e] = __fadd_rn(acc[e], __fmul_rn(kv4[e], __fdiv_rn(ex[j][e], sum[e])));
                }
            }
            // the kv have been read: the next token's kv may overwrite them
            if (more)
                prefetch_window<THREADS>(p, s_rows[i + 1], window, 1, s_win,
                                         __fadd_rn(__fadd_rn(acc[0], acc[1]), __fadd_rn(acc[2], acc[3])));
            cp_async_commit();
            finish_token<THREADS>(p, kv_shift, s_ks[i], s_prow[i], acc, s_part, s_y);
            __syncthreads();
        }
        cp_async_wait<0>();
        __syncthreads();  // every thread has read the chunk's lists before the next scan
    }
}

// ---- long windows: a cluster of CTAs per token ----------------------------------------
//
// For windows of more than 8 rows (HCA: 128).  A cluster of kSlices CTAs
// owns one writing token at a time; CTA k of the cluster owns columns
// [64k, 64k + 64), one thread per column.  Its slice of every window row
// (score and kv, 256 bytes each) is bulk-copied into shared memory in one
// round, counted by one mbarrier, and the three softmax passes run from shared
// memory in window order, each exp kept in place of its score for the
// weighted pass.  The RMSNorm's pairwise sum of squares is completed across
// the cluster: each CTA's 64-column partial (a subtree of the pairwise tree)
// goes to its shared memory, a cluster barrier, then every CTA reads the eight
// partials through distributed shared memory and adds them in the tree's
// order.  CTA k < 7 writes FP8 block k of the record; CTA 7 the RoPE tail and
// the unused scale slot.
constexpr int kSliceCols = 64;
constexpr int kSlices = kHead / kSliceCols;  // CTAs per cluster
constexpr int kColThreads = 4;                 // threads per column
constexpr int kClusterThreads = kSliceCols * kColThreads;
constexpr int kScanWarps = kClusterThreads / kWarp;  // chunks scanned per round
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Bulk-copy waits that gave up (2 s); the CTA stops copying and leaves its
// remaining rows unwritten.
__device__ unsigned int g_compress_wait_timeouts = 0;

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster; orders prior shared-memory
// accesses before the peers' later ones.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The float at `local`'s offset in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// its later bulk copies into shared memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Column c of the slice through the window, by the kColThreads threads of
// the column: thread q of it owns the contiguous rows [q W / n, (q + 1) W / n).
//  * max: part 0 folds from row 0 as the oracle does (a NaN there stays), the
//    other parts from -inf, and the parts combine in order with the same
//    strict comparison -- the oracle's first maximum (NaNs skipped);
//  * each part's exps replace its scores, then one thread of the column sums
//    them in window order;
//  * each part's kv * (exp / sum) products replace the exps, then one thread
//    sums them in window order.
// Returns the pooled value in part 0's thread (0 in the others).  Every
// thread of the CTA calls it (it holds CTA barriers).
__device__ __forceinline__ float slice_pool(float* s_sc, const float* s_kv, float* s_mx,
                                            float* s_sum, int window, int c, int q) {
    constexpr int U = 8;
    const int j0 = q * window / kColThreads, j1 = (q + 1) * window / kColThreads;
    float mx = q == 0 ? s_sc[c] : __int_as_float(0xFF800000);
#pragma unroll 8
    for (int j = (q == 0 ? 1 : j0); j < j1; ++j) {
        const float v = s_sc[j * kSliceCols + c];
        mx = v > mx ? v : mx;
    }
    s_mx[q * kSliceCols + c] = mx;
    __syncthreads();
    mx = s_mx[c];
#pragma unroll
    for (int k = 1; k < kColThreads; ++k) {
        const float v = s_mx[k * kSliceCols + c];
        mx = v > mx ? v : mx;
    }
    int j = j0;
    for (; j + U <= j1; j += U) {
        float e[U];
#pragma unroll
        for (int u = 0; u < U; u += 2)
            cw_exp2_nonpos(__fsub_rn(s_sc[(j + u) * kSliceCols + c], mx),
                           __fsub_rn(s_sc[(j + u + 1) * kSliceCols + c], mx), e[u], e[u + 1]);
#pragma unroll
        for (int u = 0; u < U; ++u) s_sc[(j + u) * kSliceCols + c] = e[u];
    }
    for (; j < j1; ++j)
        s_sc[j * kSliceCols + c] = cw_exp_nonpos(__fsub_rn(s_sc[j * kSliceCols + c], mx));
    __syncthreads();
    if (q == 0) {
        float sum = 0.0f;
#pragma unroll 8
        for (int k = 0; k < window; ++k) sum = __fadd_rn(sum, s_sc[k * kSliceCols + c]);
        s_sum[c] = sum;
    }
    __syncthreads();
    const float sum = s_sum[c];
    j = j0;
    for (; j + U <= j1; j += U) {
        float pr[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            pr[u] = __fmul_rn(s_kv[(j + u) * kSliceCols + c],
                              __fdiv_rn(s_sc[(j + u) * kSliceCols + c], sum));
#pragma unroll
        for (int u = 0; u < U; ++u) s_sc[(j + u) * kSliceCols + c] = pr[u];
    }
    for (; j < j1; ++j)
        s_sc[j * kSliceCols + c] =
            __fmul_rn(s_kv[j * kSliceCols + c], __fdiv_rn(s_sc[j * kSliceCols + c], sum));
    __syncthreads();
    float acc = 0.0f;
    if (q == 0) {
#pragma unroll 8
        for (int k = 0; k < window; ++k) acc = __fadd_rn(acc, s_sc[k * kSliceCols + c]);
    }
    return acc;
}

// Warp 0: the writing tokens among c0 .. c0 + 31 into s_list (ascending),
// their number into s_count; skips counted when `count_errors`.
__device__ __forceinline__ void scan_chunk(const CompressParams& p, int64_t c0, bool count_errors,
                                           int64_t* s_list, int* s_count) {
    const int lane = threadIdx.x & 31;
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
                    if (count_errors && p.err_count) atomicAdd(p.err_count, 1);
                } else {
                    emit = true;
                }
            }
        }
    }
    const unsigned mask = __ballot_sync(0xFFFFFFFFu, emit);
    if (emit) s_list[__popc(mask & ((1u << lane) - 1u))] = t;
    if (lane == 0) *s_count = __popc(mask);
}

// Column col0 + tid of the normalised row into token t's record: CTA k < 7
// FP8 block k (amax over the block's 64 bf16 values, the UE8M0 exponent),
// CTA 7 the GPT-J RoPE tail as bf16 and the unused scale slot.  The branch is
// uniform over the CTA.  Nothing is stored when `skip`.
__device__ __forceinline__ void slice_epilogue(const CompressParams& p, int32_t kv_shift, int64_t t,
                                               int64_t pos, uint32_t rank, float y,
                                               uint32_t* s_amax, bool owner, bool skip) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    skip = skip || !owner;  // threads 0..63 (warps 0 and 1) own the columns
    const int64_t ks = __ldg(p.kv_slots + t);
    int64_t off;
    const int64_t page = div_block(ks, p.kv_bs, kv_shift, off);
    constexpr int kTS = kNope + 2 * kRope;  // 576 data bytes per token
    uint8_t* pbase = p.kv_cache + page * p.kv_page_stride;
    uint8_t* data = pbase + off * kTS;
    uint8_t* scl = pbase + (int64_t)p.kv_bs * kTS + off * (kHead / 64);
    if ((int)rank < kNope / kSliceCols) {
        const uint32_t b = pack_bf16x2(y, 0.0f) & 0xFFFFu;
        uint32_t amb = b & 0x7FFFu;
#pragma unroll
        for (int m = 1; m < kWarp; m <<= 1) amb = max(amb, __shfl_xor_sync(0xFFFFFFFFu, amb, m));
        if (owner && lane == 0) s_amax[warp] = amb;
        __syncthreads();
        amb = max(s_amax[0], s_amax[1]);
        const float a = fmaxf(__uint_as_float(amb << 16), 1.0e-4f);
        const int e = ceil_log2_div_const(a, 0x600000u, 8);  // / 448
        const uint32_t q = cvt_e4m3x2(__fmul_rn(__uint_as_float(b << 16), exp2_int(-e)), 0.0f) & 0xFFu;
        if (!skip) {
            data[kSliceCols * rank + tid] = (uint8_t)q;
            if (tid == 0) scl[rank] = (uint8_t)min(max(e + 127, 0), 255);
        }
    } else {  // GPT-J RoPE at the group's first position: pairs (2i, 2i + 1) of the tail
        int64_t grp = pos / p.ratio;
        if (pos % p.ratio != 0 && pos < 0) grp -= 1;
        const float* cs = p.cos_sin + grp * p.ratio * p.cs_stride;
        const float other = __shfl_xor_sync(0xFFFFFFFFu, y, 1);
        const bool odd = tid & 1;
        const float ev = odd ? other : y, od = odd ? y : other;
        const int i = (tid & (kSliceCols - 1)) >> 1;
        const float c = __ldg(cs + i), sn = __ldg(cs + kRope / 2 + i);
        const float v = odd ? __fadd_rn(__fmul_rn(ev, sn), __fmul_rn(od, c))
                            : __fsub_rn(__fmul_rn(ev, c), __fmul_rn(od, sn));
        if (!skip) {
            *reinterpret_cast<uint16_t*>(data + kNope + 2 * tid) = (uint16_t)(pack_bf16x2(v, 0.0f) & 0xFFFFu);
            if (tid == 0) scl[kNope / 64] = 0;  // the unused scale slot
        }
    }
}

__global__ void __cluster_dims__(kSlices, 1, 1) __launch_bounds__(kClusterThreads)
compress_cluster_kernel(CompressParams p, int32_t kv_shift) {
    // [window][64] scores (then exps, then products), [window][64] kv
    extern __shared__ __align__(16) float s_dyn[];
    __shared__ float s_mx[kColThreads * kSliceCols];
    __shared__ float s_sum[kSliceCols];
    __shared__ float s_part[kSliceCols / kWarp];
    __shared__ float s_ssq[2];  // this CTA's partial, by token parity (read by the cluster)
    __shared__ uint32_t s_amax[kSliceCols / kWarp];
    __shared__ int s_nrows[kScanWarps];
    __shared__ int64_t s_list[kScanWarps * kWarp];
    __shared__ int s_count[kScanWarps];
    __shared__ __align__(8) uint64_t s_bar;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = tid % kSliceCols, q = tid / kSliceCols;  // column, part of the window
    const bool owner = q == 0;  // threads 0..63: the column's sums, RMSNorm and record
    const uint32_t rank = cluster_ctarank();
    const int col0 = kSliceCols * (int)rank;
    const int window = (p.overlap ? 2 : 1) * p.ratio;
    float* s_sc = s_dyn;
    float* s_kv = s_dyn + window * kSliceCols;
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();
    const int64_t nclusters = gridDim.x / kSlices;
    const int64_t cl = blockIdx.x / kSlices;
    int tok = 0;        // tokens begun by this CTA (mbarrier phase and s_ssq parity)
    bool dead = false;  // a copy wait gave up: no further copies or waits
    int dead_tok = 0;   // the token whose wait gave up
    // The cluster's chunks are cl, cl + nclusters, ...; each round, warp w
    // scans the round's w-th.  Every CTA of the cluster scans the same chunks;
    // rank 0 counts the skips.
    for (int64_t i0 = 0; (cl + i0 * nclusters) * kWarp < p.num_tokens; i0 += kScanWarps) {
        scan_chunk(p, (cl + (i0 + warp) * nclusters) * kWarp, rank == 0, s_list + warp * kWarp,
                   &s_count[warp]);
        __syncthreads();
        for (int w = 0; w < kScanWarps; ++w) {
            const int nw = s_count[w];
            for (int i = 0; i < nw; ++i, ++tok) {
                const int64_t t = s_list[w * kWarp + i];
                const int64_t pos = __ldg(p.positions + t);
                const int32_t r = __ldg(p.t2r + t);
                const int64_t base = p.base ? __ldg(p.base + r) : 0;
                // this CTA's slices of the window rows: bulk copies, absent rows filled
                int nrows = 0;
                if (!dead) {
                    fence_proxy_async_smem();
                    for (int j = tid; j < window; j += kClusterThreads) {
                        const int64_t row = window_row(p, pos, r, base, window, j);
                        if (row >= 0) {
                            const int off = (p.overlap && j >= p.ratio) ? kHead : 0;
                            const float* src = p.state + row * 2 * (int64_t)p.state_width + off + col0;
                            bulk_g2s(s_kv + j * kSliceCols, src, kSliceCols * 4, &s_bar);
                            bulk_g2s(s_sc + j * kSliceCols, src + p.state_width, kSliceCols * 4, &s_bar);
                            ++nrows;
                        } else {
                            for (int k = 0; k < kSliceCols; ++k) {
                                s_sc[j * kSliceCols + k] = -1.0e30f;
                                s_kv[j * kSliceCols + k] = 0.0f;
                            }
                        }
                    }
                }
                nrows = __reduce_add_sync(0xFFFFFFFFu, nrows);
                if (lane == 0) s_nrows[warp] = nrows;
                __syncthreads();
                if (!dead && tid == 0) {
                    int total = 0;
                    for (int k = 0; k < kScanWarps; ++k) total += s_nrows[k];
                    mbar_arrive_expect_tx(&s_bar, (uint32_t)total * 2u * kSliceCols * 4u);
                }
                const bool landed =
                    dead ? false : mbar_wait_bounded(&s_bar, (uint32_t)(tok & 1), kWaitLimitNs);
                if (!dead && !__syncthreads_and(landed)) {
                    if (tid == 0) atomicAdd(&g_compress_wait_timeouts, 1u);
                    dead = true;
                    dead_tok = tok;
                }
                // pooling, then this CTA's part of the pairwise sum of squares
                const float acc = dead ? 0.0f : slice_pool(s_sc, s_kv, s_mx, s_sum, window, c, q);
                float ssq = __fmul_rn(acc, acc);
#pragma unroll
                for (int m = 1; m < kWarp; m <<= 1)
                    ssq = __fadd_rn(ssq, __shfl_xor_sync(0xFFFFFFFFu, ssq, m));
                if (owner && lane == 0) s_part[warp] = ssq;
                __syncthreads();
                if (tid == 0) s_ssq[tok & 1] = __fadd_rn(s_part[0], s_part[1]);
                cluster_sync_all();
                float part[kSlices];
#pragma unroll
                for (int k = 0; k < kSlices; ++k) part[k] = ld_cluster_f32(&s_ssq[tok & 1], (uint32_t)k);
#pragma unroll
                for (int h = kSlices / 2; h >= 1; h >>= 1)
#pragma unroll
                    for (int k = 0; k < h; ++k) part[k] = __fadd_rn(part[2 * k], part[2 * k + 1]);
                const float variance = __fmul_rn(part[0], 1.0f / kHead);  // exact: a power of two
                const float rr = __frcp_rn(__fsqrt_rn(__fadd_rn(variance, p.eps)));
                const float y = __fmul_rn(__fmul_rn(acc, rr), __ldg(p.weight + col0 + c));
                slice_epilogue(p, kv_shift, t, pos, rank, y, s_amax, owner, dead);
                __syncthreads();  // the slices are read before the next token's copies
            }
        }
        __syncthreads();  // every thread has read s_count / s_list before the next scan
    }
    // no CTA leaves while a peer may read its partial; copies of a CTA whose
    // wait gave up are waited for (bounded) before it retires
    cluster_sync_all();
    if (dead && tid == 0) mbar_wait_bounded(&s_bar, (uint32_t)(dead_tok & 1), kWaitLimitNs);
}

}  // namespace

cudaError_t read_compress_wait_timeouts(uint32_t* count) {
    return cudaMemcpyFromSymbol(count, g_compress_wait_timeouts, sizeof(uint32_t));
}

cudaError_t launch_save_compressor_state(const SaveStateParams& p, cudaStream_t stream) {
    const int64_t blocks = (p.num_tokens * kWarp + kThreads - 1) / kThreads;
    return launch_pdl(save_state_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream, p);
}

cudaError_t launch_compress_kv_insert(const CompressParams& p, cudaStream_t stream) {
    const int window = (p.overlap ? 2 : 1) * p.ratio;
    const int32_t shift = log2_if_pow2(p.kv_bs);
    const int64_t chunks = (p.num_tokens + kWarp - 1) / kWarp;
    if (window <= 8) {
        // 32-token chunks (16-token chunks, which fill every resident CTA
        // slot, measured slower: twice the scans)
        constexpr int kChunk = 32;
        auto kern = compress_kernel<128, kChunk>;
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 128, 0) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        const int64_t nchunks = (p.num_tokens + kChunk - 1) / kChunk;
        const int64_t full = (int64_t)sm_count() * per_sm;
        return launch_pdl(kern, dim3((unsigned)(nchunks < full ? nchunks : full)), dim3(128), 0,
                          stream, p, shift);
    }
    // longer windows: clusters of kSlices CTAs, as many as can be resident
    auto kern = compress_cluster_kernel;
    const size_t smem = (size_t)window * kSliceCols * 2 * sizeof(float);
    static std::atomic<uint64_t> limit_set{0};
    const cudaError_t e = set_smem_limit_per_device(
        kern, (int)(kMaxWindow * kSliceCols * 2 * sizeof(float)), limit_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kSlices);
    cfg.blockDim = dim3(kClusterThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess || max_clusters < 1)
        max_clusters = 1;
    const int64_t per_round = (int64_t)kScanWarps;
    const int64_t want = (chunks + per_round - 1) / per_round;
    const int64_t clusters = want < max_clusters ? want : max_clusters;
    return launch_pdl(kern, dim3((unsigned)(clusters * kSlices)), dim3(kClusterThreads), smem, stream,
                      p, shift);
}

}  // namespace psk
