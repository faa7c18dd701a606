// index_build.cu -- sparse-index builders.
//
// Fused window + top-k build: vLLM deepseek_v41 ops,
// build_flashinfer_mixed_sparse_indices (TokenSpeed's combine_topk_swa_indices
// step).  Top-k mapping alone: vLLM compute_global_topk_indices_and_lens.
// Token positions follow TokenSpeed backends/deepseek_v4.py,
// _decode_positions_from_metadata.
//
// Design (integer, HBM-bound, latency-sensitive at decode sizes):
//  * A warp slice owns one token row; lanes walk the row in 16-byte quads
//    (4 int32 columns) when every row starts on a 16-byte boundary, else one
//    column at a time.  Top-k quads are one int4 load and one int4 store.
//  * Window columns are computed, not loaded: column c is position lo + c.
//  * The block-table rows of a CTA whose tokens all belong to one request are
//    staged in shared memory once, so every slot look-up (random top-k ones
//    and the window's) hits shared memory (the shared-memory block-table tiles).
//  * Two memory round trips before any output: token -> request indices and
//    the first top-k quads, then the request's metadata together with the
//    table rows.
//  * lens is a warp reduction (__reduce_add_sync) of per-lane valid counts,
//    combined across the warps of a token in shared memory when a token is
//    split over several warps (small batches: every SM gets work).
#include <algorithm>
#include <climits>

#include "index_build.h"
#include "psk_common.cuh"

namespace psk {
namespace {

// Launch-shape constants (overridable at build time for tuning sweeps).
#ifndef PSK_INDEX_BATCH
#define PSK_INDEX_BATCH 4
#endif
#ifndef PSK_WS_INDEX_BATCH
#define PSK_WS_INDEX_BATCH 4
#endif
#ifndef PSK_INDEX_MAX_PASSES
#define PSK_INDEX_MAX_PASSES 1
#endif
#ifndef PSK_WS_INDEX_MAX_PASSES
#define PSK_WS_INDEX_MAX_PASSES 2
#endif
#ifndef PSK_INDEX_SB_UNROLL
#define PSK_INDEX_SB_UNROLL 1
#endif
#ifndef PSK_INDEX_WARPS_PER_SM
#define PSK_INDEX_WARPS_PER_SM 16  // split a token over warps below this many token-warps per SM
#endif
#ifndef PSK_INDEX_MIN_CTAS
#define PSK_INDEX_MIN_CTAS 3
#endif
// Resident CTAs per SM asked of the staged-row builders (launch bounds).  Four
// by default.  The top-k map also has a build for 5 (46 registers instead of 53,
// no spills), taken when the grid exceeds one wave at 4 per SM: on the
// 16384-token prefill (3.4 waves) it runs 19.9 us against 20.8; inside one wave
// (the 4352-token mixed batch) the 53-register build is faster (14.3 us against
// 16.3).  The fused window + top-k build stays at 4 (at 5 it spills and gains
// nothing, at 3 or 6 it slows from 22.5 to 24.6 us).
#ifndef PSK_INDEX_TMA_MIN_CTAS
#define PSK_INDEX_TMA_MIN_CTAS 4
#endif
#ifndef PSK_INDEX_TMA_MIN_CTAS_WIDE
#define PSK_INDEX_TMA_MIN_CTAS_WIDE 5
#endif

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / kWarp;
constexpr int kSbUnroll = PSK_INDEX_SB_UNROLL;
constexpr int kMaxStagedEntries = 4096;  // 16 KB of int32 page ids per staged row
constexpr int kMaxTopkStageBytes = 64 * 1024;  // top-k rows of one CTA in shared memory
constexpr int kTopkBars = 16;                  // staged top-k rows (tokens) per CTA at most
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Waits on the top-k staging barrier that gave up (2 s without the copies
// landing); the rows of that CTA are left unwritten.
__device__ unsigned int g_index_wait_timeouts = 0;

struct TableRow {
    const int32_t* row;  // global row, or shared copy
    int32_t width;
    int32_t base;
    int32_t bs;
    int32_t shift;  // log2(bs) (POW2 kernels)
    int32_t maxp;   // INT32_MAX / bs: largest page whose slots can fit in int32
    int32_t maxrem; // INT32_MAX % bs
};

// Slot of logical position p (0 <= p <= INT32_MAX) through one block-table
// row, or -1: logical page p / bs - base outside [0, width), a negative page,
// or a slot beyond INT32_MAX.  All 32-bit: q - base is formed modulo 2^32 and
// tested as unsigned against width; it wraps only when the true logical page
// is >= 2^31 (q >= 0, base >= -2^31), and then the wrapped value is negative,
// i.e. rejected, as the true one would be.  POW2 (bs = 2^shift): a page
// p <= maxp = INT32_MAX >> shift gives page * bs + rem <= INT32_MAX for every
// rem < bs, so one unsigned compare rejects both negative and too-large pages.
template <bool SHARED, bool POW2>
__device__ __forceinline__ int32_t map_slot(const TableRow& tr, int32_t p) {
    int32_t q, rem;
    if (POW2) {
        q = p >> tr.shift;
        rem = p & (tr.bs - 1);
    } else {
        q = (int32_t)((uint32_t)p / (uint32_t)tr.bs);
        rem = p - q * tr.bs;
    }
    const uint32_t lp = (uint32_t)q - (uint32_t)tr.base;
    if (lp >= (uint32_t)tr.width) return -1;
    const int32_t page = SHARED ? tr.row[lp] : __ldg(tr.row + lp);
    if (POW2) return (uint32_t)page > (uint32_t)tr.maxp ? -1 : ((page << tr.shift) | rem);
    if ((uint32_t)page > (uint32_t)tr.maxp || (page == tr.maxp && rem > tr.maxrem)) return -1;
    return page * tr.bs + rem;
}

// The same rule for any position p >= 0 (window positions past INT32_MAX,
// which only metadata whose tokens lie outside their request's query range
// can produce).
__device__ __forceinline__ int32_t map_slot_wide(const TableRow& tr, int64_t p) {
    const int64_t q = p / tr.bs;
    const int64_t lp = q - tr.base;
    if (lp < 0 || lp >= tr.width) return -1;
    const int32_t page = __ldg(tr.row + lp);  // a global row
    if (page < 0) return -1;
    const int64_t s = (int64_t)page * tr.bs + (p - q * tr.bs);
    return s > 0x7FFFFFFFll ? -1 : (int32_t)s;
}

// Per-token values that depend on its request (second memory round trip).
// Window columns c < nwin hold positions lo + c <= pos.
struct TokMeta {
    int32_t r;
    bool ok;
    bool wide;  // pos > INT32_MAX: window slots through map_slot_wide
    int32_t nwin;
    int64_t lo;
    int32_t swa_base, comp_base;
};

template <bool HAS_SWA>
__device__ __forceinline__ TokMeta load_meta(const IndexParams& p, int64_t t, int32_t r) {
    TokMeta m;
    m.r = r;
    m.ok = (p.valid == nullptr || __ldg(p.valid + t) != 0) && r >= 0 && r < p.num_reqs;
    m.lo = 0;
    m.nwin = 0;
    m.wide = false;
    m.swa_base = m.comp_base = 0;
    if (!m.ok) return m;
    m.comp_base = p.comp_base ? __ldg(p.comp_base + r) : 0;
    if (HAS_SWA) {
        m.swa_base = p.swa_base ? __ldg(p.swa_base + r) : 0;
        const int64_t qs = __ldg(p.qsl + r);
        const int64_t qe = __ldg(p.qsl + r + 1);
        const int64_t pos = (int64_t)__ldg(p.seq_lens + r) - (qe - qs) + (t - qs);
        int64_t lo = pos - p.window + 1;
        const int64_t rs = p.replay ? (int64_t)__ldg(p.replay + r) : 0;
        if (rs > lo) lo = rs;
        if (lo < 0) lo = 0;
        m.lo = lo;
        const int64_t n = pos - lo + 1;  // <= window
        m.nwin = n > 0 ? (int32_t)n : 0;
        m.wide = pos > 0x7FFFFFFFll;
    }
    return m;
}

// Loads the top-k quad that starts at output column c0 (-1 past topk).
__device__ __forceinline__ int4 load_topk_quad(const IndexParams& p, const int32_t* tk, int j0) {
    if (j0 + 3 < p.topk) return __ldg(reinterpret_cast<const int4*>(tk + j0));
    return make_int4(j0 < p.topk ? __ldg(tk + j0) : -1, j0 + 1 < p.topk ? __ldg(tk + j0 + 1) : -1,
                     j0 + 2 < p.topk ? __ldg(tk + j0 + 2) : -1, -1);
}

// Token t's row when its window positions pass INT32_MAX: one column per
// lane step, window slots through the 64-bit rule, both rows in global memory.
template <bool POW2>
__device__ __noinline__ int build_row_wide(const IndexParams& p, int64_t t, const TokMeta& m,
                                           int first, int stride, TableRow swa, TableRow comp) {
    int32_t* out = p.out + t * p.out_stride;
    const int32_t* tk = p.topk_local + t * p.topk_stride;
    swa.row = p.swa_bt + (int64_t)m.r * p.swa_stride;
    comp.row = p.comp_bt + (int64_t)m.r * p.comp_stride;
    int cnt = 0;
    for (int c = first; c < p.out_cols; c += stride) {
        int v;
        if (c < p.window) {
            v = c < m.nwin ? map_slot_wide(swa, m.lo + c) : -1;
        } else {
            const int j = c - p.window;
            const int l = j < p.topk ? __ldg(tk + j) : -1;
            v = l >= 0 ? map_slot<false, POW2>(comp, l) : -1;
        }
        cnt += v >= 0;
        out[c] = v;
    }
    return cnt;
}

// Writes token t's row and returns this lane's count of valid entries.
// `pre` holds the lane's first batch of top-k quads, loaded in advance (VEC).
// STAGED: the token's table rows are in shared memory (else read through L1).
template <bool HAS_SWA, bool VEC, bool POW2, bool STAGED>
__device__ __forceinline__ int build_row(const IndexParams& p, int64_t t, const TokMeta& m,
                                         int first, int stride, const int4 (&pre)[PSK_INDEX_BATCH],
                                         const int32_t* s_swa, const int32_t* s_comp) {
    int32_t* out = p.out + t * p.out_stride;
    if (!m.ok) {
        if (VEC) {
            const int nq = (p.out_cols + 3) / 4;
            for (int q = first; q < nq; q += stride) {
                const int c0 = 4 * q;
                if (c0 + 3 < p.out_cols) {
                    *reinterpret_cast<int4*>(out + c0) = make_int4(-1, -1, -1, -1);
                } else {
                    for (int c = c0; c < p.out_cols; ++c) out[c] = -1;
                }
            }
        } else {
            for (int c = first; c < p.out_cols; c += stride) out[c] = -1;
        }
        return 0;
    }
    TableRow comp;
    comp.row = STAGED ? s_comp : p.comp_bt + (int64_t)m.r * p.comp_stride;
    comp.width = p.comp_width;
    comp.base = m.comp_base;
    comp.bs = p.comp_bs;
    comp.shift = p.comp_shift;
    comp.maxp = p.comp_maxp;
    comp.maxrem = p.comp_maxrem;
    TableRow swa;
    if (HAS_SWA) {
        swa.row = STAGED ? s_swa : p.swa_bt + (int64_t)m.r * p.swa_stride;
        swa.width = p.swa_width;
        swa.base = m.swa_base;
        swa.bs = p.swa_bs;
        swa.shift = p.swa_shift;
        swa.maxp = p.swa_maxp;
        swa.maxrem = p.swa_maxrem;
    }
    const int32_t* tk = p.topk_local + t * p.topk_stride;
    const int W = HAS_SWA ? p.window : 0;
    if (HAS_SWA && m.wide) return build_row_wide<POW2>(p, t, m, first, stride, swa, comp);

    int cnt = 0;
    if (VEC) {
        // Quads are processed in batches of kBatch per lane: every top-k load
        // of a batch is issued before any of them is used.
        constexpr int kBatch = PSK_INDEX_BATCH;
        const int nq = (p.out_cols + 3) / 4;
        for (int qb = first; qb < nq; qb += kBatch * stride) {
            int4 L[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int q = qb + u * stride;
                const int c0 = 4 * q;
                L[u] = make_int4(-1, -1, -1, -1);
                if (qb == first) L[u] = pre[u];
                else if (q < nq && c0 >= W) L[u] = load_topk_quad(p, tk, c0 - W);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int q = qb + u * stride;
                if (q >= nq) break;
                const int c0 = 4 * q;
                int v[4];
                if (HAS_SWA && c0 < W) {
                    const int32_t lo = (int32_t)m.lo;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        v[e] = c0 + e < m.nwin ? map_slot<STAGED, POW2>(swa, lo + c0 + e) : -1;
                } else {
                    const int4 w = L[u];
                    v[0] = w.x >= 0 ? map_slot<STAGED, POW2>(comp, w.x) : -1;
                    v[1] = w.y >= 0 ? map_slot<STAGED, POW2>(comp, w.y) : -1;
                    v[2] = w.z >= 0 ? map_slot<STAGED, POW2>(comp, w.z) : -1;
                    v[3] = w.w >= 0 ? map_slot<STAGED, POW2>(comp, w.w) : -1;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) cnt += v[e] >= 0;
                if (c0 + 3 < p.out_cols) {
                    *reinterpret_cast<int4*>(out + c0) = make_int4(v[0], v[1], v[2], v[3]);
                } else {
                    out[c0] = v[0];
                    if (c0 + 1 < p.out_cols) out[c0 + 1] = v[1];
                    if (c0 + 2 < p.out_cols) out[c0 + 2] = v[2];
                }
            }
        }
    } else {
        for (int c = first; c < p.out_cols; c += stride) {
            int v;
            if (HAS_SWA && c < W) {
                v = c < m.nwin ? map_slot<STAGED, POW2>(swa, (int32_t)m.lo + c) : -1;
            } else {
                const int j = c - W;
                const int l = j < p.topk ? __ldg(tk + j) : -1;
                v = l >= 0 ? map_slot<STAGED, POW2>(comp, l) : -1;
            }
            cnt += v >= 0;
            out[c] = v;
        }
    }
    return cnt;
}

// Token t's row from its top-k row staged in shared memory (s_row; the TMA
// kernels: VEC layout, topk % 4 == 0, so a quad is all top-k or all past it).
template <bool HAS_SWA, bool POW2, bool STAGED>
__device__ __forceinline__ int build_row_smem(const IndexParams& p, int64_t t, const TokMeta& m,
                                              int first, int stride, const int32_t* s_row,
                                              const int32_t* s_swa, const int32_t* s_comp) {
    int32_t* out = p.out + t * p.out_stride;
    const int nq = p.out_cols / 4;
    if (!m.ok) {
        for (int q = first; q < nq; q += stride)
            *reinterpret_cast<int4*>(out + 4 * q) = make_int4(-1, -1, -1, -1);
        return 0;
    }
    TableRow comp;
    comp.row = STAGED ? s_comp : p.comp_bt + (int64_t)m.r * p.comp_stride;
    comp.width = p.comp_width;
    comp.base = m.comp_base;
    comp.bs = p.comp_bs;
    comp.shift = p.comp_shift;
    comp.maxp = p.comp_maxp;
    comp.maxrem = p.comp_maxrem;
    TableRow swa;
    if (HAS_SWA) {
        swa.row = STAGED ? s_swa : p.swa_bt + (int64_t)m.r * p.swa_stride;
        swa.width = p.swa_width;
        swa.base = m.swa_base;
        swa.bs = p.swa_bs;
        swa.shift = p.swa_shift;
        swa.maxp = p.swa_maxp;
        swa.maxrem = p.swa_maxrem;
    }
    const int W = HAS_SWA ? p.window : 0;
    if (HAS_SWA && m.wide) return build_row_wide<POW2>(p, t, m, first, stride, swa, comp);
    int cnt = 0;
#pragma unroll 2
    for (int q = first; q < nq; q += stride) {
        const int c0 = 4 * q;
        int v[4];
        if (HAS_SWA && c0 < W) {
            const int32_t lo = (int32_t)m.lo;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                v[e] = c0 + e < m.nwin ? map_slot<STAGED, POW2>(swa, lo + c0 + e) : -1;
        } else {
            const int j0 = c0 - W;
            const int4 w = j0 < p.topk ? *reinterpret_cast<const int4*>(s_row + j0)
                                       : make_int4(-1, -1, -1, -1);
            v[0] = w.x >= 0 ? map_slot<STAGED, POW2>(comp, w.x) : -1;
            v[1] = w.y >= 0 ? map_slot<STAGED, POW2>(comp, w.y) : -1;
            v[2] = w.z >= 0 ? map_slot<STAGED, POW2>(comp, w.z) : -1;
            v[3] = w.w >= 0 ? map_slot<STAGED, POW2>(comp, w.w) : -1;
        }
        cnt += (v[0] >= 0) + (v[1] >= 0) + (v[2] >= 0) + (v[3] >= 0);
        *reinterpret_cast<int4*>(out + c0) = make_int4(v[0], v[1], v[2], v[3]);
    }
    return cnt;
}

// ---- slot-base tables (power-of-two pages, the CTA's request staged) ---------------
//
// A staged table row held as slot bases: entry i is page_i << shift, or -1
// when page_i is negative or its slots would pass INT32_MAX (page > maxp), and
// one more entry, at index width, is -1.  A position p then maps to
// base[i] | (p & (bs - 1)) with i = (p >> shift) - table_base when p lies in
// the row's position range, else to base[width] = -1: -1 | rem stays -1.
__device__ __forceinline__ void stage_slot_bases(int32_t* dst, const int32_t* src, int n,
                                                 int shift, int32_t maxp) {
    for (int i0 = threadIdx.x; i0 <= n; i0 += 4 * kThreads) {
        int32_t v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kThreads;
            v[u] = i < n ? __ldg(src + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kThreads;
            if (i <= n) dst[i] = (uint32_t)v[u] > (uint32_t)maxp ? -1 : (v[u] << shift);
        }
    }
}

// The positions [lo, lo + span) that one staged row maps: its pages'
// positions, clipped to [0, 2^31) and to [clip_lo, clip_hi).
struct SbRange {
    uint32_t lo;    // first mapped position
    uint32_t span;  // number of mapped positions (0: none)
    int32_t base;   // table base offset (logical page of entry 0)
};

__device__ __forceinline__ SbRange sb_range(int32_t base, int32_t width, int shift,
                                            int64_t clip_lo, int64_t clip_hi) {
    int64_t lo = (int64_t)base << shift;
    int64_t hi = lo + ((int64_t)width << shift);
    if (lo < clip_lo) lo = clip_lo;
    if (hi > clip_hi) hi = clip_hi;
    if (lo < 0) lo = 0;
    if (hi > 0x80000000ll) hi = 0x80000000ll;
    SbRange r;
    r.lo = hi > lo ? (uint32_t)lo : 0u;
    r.span = hi > lo ? (uint32_t)(hi - lo) : 0u;
    r.base = base;
    return r;
}

// Slot of position p through a slot-base row (see above): one unsigned range
// test, one shared load, one OR.  Positions below lo (negative ones included)
// wrap to >= span.  In range, p >= 0 and (p >> shift) - base lies in [0, width).
__device__ __forceinline__ int32_t sb_slot(const int32_t* sb, const SbRange& r, int width,
                                           int shift, int32_t mask, int32_t p) {
    const bool in = (uint32_t)p - r.lo < r.span;
    const int i = in ? (int)(((uint32_t)p >> shift) - (uint32_t)r.base) : width;
    return sb[i] | (p & mask);
}

// Token t's row (window columns then top-k columns) through the CTA's staged
// slot-base rows; the top-k row is in shared memory (s_row).  The same values
// as build_row_smem with the tables staged.
template <bool HAS_SWA>
__device__ __forceinline__ int build_row_sb(const IndexParams& p, int64_t t, const TokMeta& m,
                                            int first, int stride, const int32_t* s_row,
                                            const int32_t* s_swa, const int32_t* s_comp) {
    int32_t* out = p.out + t * p.out_stride;
    const int nq = p.out_cols / 4;
    if (!m.ok) {
        for (int q = first; q < nq; q += stride)
            *reinterpret_cast<int4*>(out + 4 * q) = make_int4(-1, -1, -1, -1);
        return 0;
    }
    const int W = HAS_SWA ? p.window : 0;
    const int cshift = p.comp_shift;
    const int32_t cmask = p.comp_bs - 1;
    const SbRange cr = sb_range(m.comp_base, p.comp_width, cshift, 0, 0x80000000ll);
    SbRange wr{};
    int sshift = 0;
    int32_t smask = 0;
    if (HAS_SWA) {
        sshift = p.swa_shift;
        smask = p.swa_bs - 1;
        // window column c holds position lo + c for c < nwin
        wr = sb_range(m.swa_base, p.swa_width, sshift, m.lo, m.lo + m.nwin);
    }
    int invalid = 0;  // minus the count of valid entries written by this lane
    int cols = 0;
#pragma unroll kSbUnroll
    for (int q = first; q < nq; q += stride) {
        const int c0 = 4 * q;
        int v[4];
        if (HAS_SWA && c0 < W) {
            // m.lo <= INT32_MAX (not a wide token); columns past nwin wrap out of range
            const uint32_t pos0 = (uint32_t)m.lo + (uint32_t)c0;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                v[e] = sb_slot(s_swa, wr, p.swa_width, sshift, smask, (int32_t)(pos0 + (uint32_t)e));
        } else {
            const int4 w = *reinterpret_cast<const int4*>(s_row + (c0 - W));
            v[0] = sb_slot(s_comp, cr, p.comp_width, cshift, cmask, w.x);
            v[1] = sb_slot(s_comp, cr, p.comp_width, cshift, cmask, w.y);
            v[2] = sb_slot(s_comp, cr, p.comp_width, cshift, cmask, w.z);
            v[3] = sb_slot(s_comp, cr, p.comp_width, cshift, cmask, w.w);
        }
        invalid += (v[0] >> 31) + (v[1] >> 31) + (v[2] >> 31) + (v[3] >> 31);
        cols += 4;
        *reinterpret_cast<int4*>(out + c0) = make_int4(v[0], v[1], v[2], v[3]);
    }
    return cols + invalid;
}

// Thread 0 of the CTA: one bulk copy per token row t0..t1-1 of topk_local
// into `dst` (rows of `words` int32), all completing on `bar`.  Returns the
// bytes expected.  Every address and size is a multiple of 16 bytes (16-byte
// aligned topk_local, topk_stride and topk multiples of 4).
__device__ __forceinline__ void stage_topk_rows(int32_t* dst, const int32_t* topk_local,
                                                int64_t topk_stride, int words, int64_t t0,
                                                int64_t t1, uint64_t* bar) {
    const uint32_t bytes = (uint32_t)words * 4u;
    mbar_arrive_expect_tx(bar, bytes * (uint32_t)(t1 - t0));
    for (int64_t t = t0; t < t1; ++t)
        bulk_g2s(dst + (t - t0) * words, topk_local + t * topk_stride, bytes, bar);
}

// The same with one barrier per token row: row t - t0 completes on
// bars[t - t0], so each token's warps start as soon as their own row lands.
__device__ __forceinline__ void stage_topk_rows_each(int32_t* dst, const int32_t* topk_local,
                                                     int64_t topk_stride, int words, int64_t t0,
                                                     int64_t t1, uint64_t* bars) {
    const uint32_t bytes = (uint32_t)words * 4u;
    for (int64_t t = t0; t < t1; ++t) {
        mbar_arrive_expect_tx(&bars[t - t0], bytes);
        bulk_g2s(dst + (t - t0) * words, topk_local + t * topk_stride, bytes, &bars[t - t0]);
    }
}

// Loads the lane's first batch of top-k quads of token t (depends on t only).
template <bool VEC>
__device__ __forceinline__ void load_first_batch(const IndexParams& p, int64_t t, int64_t t1,
                                                 int first, int stride, int W,
                                                 int4 (&pre)[PSK_INDEX_BATCH]) {
#pragma unroll
    for (int u = 0; u < PSK_INDEX_BATCH; ++u) {
        const int c0 = 4 * (first + u * stride);
        pre[u] = make_int4(-1, -1, -1, -1);
        if (VEC && t < t1 && c0 >= W && c0 < p.out_cols)
            pre[u] = load_topk_quad(p, p.topk_local + t * p.topk_stride, c0 - W);
    }
}

// Copies `n` table entries to shared memory, 4 loads in flight per thread.
__device__ __forceinline__ void stage_row(int32_t* dst, const int32_t* src, int n) {
    for (int i0 = threadIdx.x; i0 < n; i0 += 4 * kThreads) {
        int32_t v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kThreads;
            v[u] = i < n ? __ldg(src + i) : 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kThreads;
            if (i < n) dst[i] = v[u];
        }
    }
}

template <bool HAS_SWA, bool VEC, bool POW2, bool TMA, int MINB = PSK_INDEX_TMA_MIN_CTAS>
__global__ void __launch_bounds__(kThreads, TMA ? MINB : PSK_INDEX_MIN_CTAS)
index_build_kernel(IndexParams p) {
    // Dynamic shared memory: [TMA: tokens_per_cta top-k rows][compressed
    // table row + 1][SWA table row + 1].  With staged top-k rows and
    // power-of-two pages the table rows are held as slot bases.
    constexpr bool SB = TMA && POW2;
    extern __shared__ __align__(16) int32_t s_dyn[];
    __shared__ int s_cnt[kWarps];
    __shared__ __align__(8) uint64_t s_bar[kTopkBars];  // one per staged token row
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t t0 = (int64_t)blockIdx.x * p.tokens_per_cta;
    int64_t t1 = t0 + p.tokens_per_cta;
    if (t1 > p.num_tokens) t1 = p.num_tokens;
    const int wpt = p.warps_per_token;
    const int tpp = kWarps / wpt;  // tokens per pass
    const int tslot = warp / wpt;
    const int slice = warp % wpt;
    const int first = slice * kWarp + lane;
    const int stride = wpt * kWarp;
    const int W = HAS_SWA ? p.window : 0;
    const bool copy_topk = TMA && p.topk > 0;
    int32_t* s_topk = s_dyn;
    int32_t* s_comp = s_dyn + (TMA ? p.tokens_per_cta * p.topk : 0);
    int32_t* s_swa = s_comp + p.stage_comp + 1;
    if (TMA && threadIdx.x == 0) {
        for (int i = 0; i < kTopkBars; ++i) mbar_init(&s_bar[i], 1);
        mbar_fence_init();
    }
    if (TMA) __syncthreads();
    // Every input may come from the previous kernel on the stream: nothing
    // global is read before its grid is done.
    pdl_wait();
    pdl_launch_dependents();

    // First memory round trip: loads that depend only on token indices (TMA: the CTA's
    // top-k rows, in flight while the metadata arrives).
    if (copy_topk && threadIdx.x == 0)
        stage_topk_rows_each(s_topk, p.topk_local, p.topk_stride, p.topk, t0, t1, s_bar);
    const int32_t r0 = __ldg(p.t2r + t0);
    const int32_t r1 = __ldg(p.t2r + t1 - 1);
    const int64_t tf = t0 + tslot;  // this warp's first token
    int32_t rf = -1;
    int4 pre[PSK_INDEX_BATCH];
    if (tf < t1) rf = __ldg(p.t2r + tf);
    if (!TMA) load_first_batch<VEC>(p, tf, t1, first, stride, W, pre);
    // Second round trip: the first token's request metadata and, when the tile is one
    // request, its block-table rows into shared memory.
    TokMeta mf;
    if (tf < t1) mf = load_meta<HAS_SWA>(p, tf, rf);
    // Stage only when every row the tile needs fits (p.stage_* > 0 exactly then).
    const bool fits = p.stage_comp > 0 && (!HAS_SWA || p.stage_swa > 0);
    const int32_t staged = (fits && r0 == r1 && r0 >= 0 && r0 < p.num_reqs) ? r0 : -1;
    if (staged >= 0 && SB) {
        stage_slot_bases(s_comp, p.comp_bt + (int64_t)staged * p.comp_stride, p.stage_comp,
                         p.comp_shift, p.comp_maxp);
        if (HAS_SWA)
            stage_slot_bases(s_swa, p.swa_bt + (int64_t)staged * p.swa_stride, p.stage_swa,
                             p.swa_shift, p.swa_maxp);
    } else if (staged >= 0) {
        stage_row(s_comp, p.comp_bt + (int64_t)staged * p.comp_stride, p.stage_comp);
        if (HAS_SWA) stage_row(s_swa, p.swa_bt + (int64_t)staged * p.swa_stride, p.stage_swa);
    }
    __syncthreads();

    for (int64_t tb = t0; tb < t1; tb += tpp) {
        const int64_t t = tb + tslot;
        int cnt = 0;
        bool rows_ok = true;  // this token's staged top-k row landed
        if (copy_topk && t < t1) {
            rows_ok = mbar_wait_bounded(&s_bar[t - t0], 0, kWaitLimitNs);
            if (!rows_ok && lane == 0) atomicAdd(&g_index_wait_timeouts, 1u);
        }
        if (t < t1 && rows_ok) {
            TokMeta m;
            if (tb == t0) {
                m = mf;
            } else {
                m = load_meta<HAS_SWA>(p, t, __ldg(p.t2r + t));
                if (!TMA) load_first_batch<VEC>(p, t, t1, first, stride, W, pre);
            }
            if (TMA) {
                const int32_t* s_row = s_topk + (t - t0) * p.topk;
                // (a wide token's row reads global tables only)
                if (staged >= 0 && m.r == staged && SB && !m.wide)
                    cnt = build_row_sb<HAS_SWA>(p, t, m, first, stride, s_row, s_swa, s_comp);
                else if (staged >= 0 && m.r == staged)
                    cnt = build_row_smem<HAS_SWA, POW2, true>(p, t, m, first, stride, s_row, s_swa, s_comp);
                else
                    cnt = build_row_smem<HAS_SWA, POW2, false>(p, t, m, first, stride, s_row, s_swa, s_comp);
            } else {
                if (staged >= 0 && m.r == staged)
                    cnt = build_row<HAS_SWA, VEC, POW2, true>(p, t, m, first, stride, pre, s_swa, s_comp);
                else
                    cnt = build_row<HAS_SWA, VEC, POW2, false>(p, t, m, first, stride, pre, s_swa, s_comp);
            }
        }
        cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
        if (wpt == 1) {
            if (lane == 0 && t < t1 && rows_ok) p.lens[t] = cnt;
        } else {
            if (lane == 0) s_cnt[warp] = cnt;
            __syncthreads();
            if (slice == 0 && lane == 0 && t < t1 && rows_ok) {
                int sum = 0;
                for (int i = 0; i < wpt; ++i) sum += s_cnt[warp + i];
                p.lens[t] = sum;
            }
            __syncthreads();
        }
    }
    // No CTA retires with copies still landing in its shared memory: thread 0
    // waits (bounded) on every row's barrier -- at once for rows that landed,
    // each used for one phase only.
    if (copy_topk && threadIdx.x == 0)
        for (int64_t t = t0; t < t1; ++t) mbar_wait_bounded(&s_bar[t - t0], 0, kWaitLimitNs);
}

// ---- workspace-relative form ------------------------------------------------------
//
// TokenSpeed's combine_topk_swa_indices as the prefill workspace path calls it
// (backends/deepseek_v4.py, _prefill_workspace): request r's rows start at
// r * workspace_width, compressed entries at rows 0.., the gathered window
// positions g0 = seq - gather_len .. seq - 1 at rows compressed_base...  No
// table look-ups: every column is arithmetic on the token's metadata.
// A token's metadata, and both column rules in 32-bit form.  Window column
// c < W holds position ps = lo + c: row rbase + compressed_base + (ps - g0)
// when g0 <= ps <= pos, i.e. row wb + c for c in [wc_lo, wc_lo + wc_n) (the
// range also clipped to rows <= INT32_MAX, which become -1).  Top-k column
// with entry l: row rbase + l when 0 <= l < lc, i.e. for (uint32)l < tk_n (the
// bound also clipped to rows <= INT32_MAX).  Both are worked out once per
// token in 64-bit arithmetic (ws_forms).
struct WsMeta {
    bool ok;
    int64_t pos, lo, g0, lc, rbase;
    int32_t wc_lo, wb, rb;
    uint32_t wc_n, tk_n;
};

__device__ __forceinline__ void ws_forms(const WorkspaceIndexParams& p, WsMeta& m) {
    m.wc_lo = m.wb = m.rb = 0;
    m.wc_n = m.tk_n = 0u;
    if (!m.ok) return;
    const int64_t base = m.rbase + p.compressed_base - m.g0 + m.lo;  // row of column 0
    const int64_t clo = m.g0 > m.lo ? m.g0 - m.lo : 0;
    int64_t chi = (int64_t)p.window - 1;
    if (m.pos - m.lo < chi) chi = m.pos - m.lo;
    if (0x7FFFFFFFll - base < chi) chi = 0x7FFFFFFFll - base;
    if (chi >= clo) {
        m.wc_lo = (int32_t)clo;
        m.wc_n = (uint32_t)(chi - clo + 1);
        m.wb = (int32_t)(uint32_t)(uint64_t)base;  // base + c is exact modulo 2^32
    }
    int64_t hi = m.lc;
    if (0x80000000ll - m.rbase < hi) hi = 0x80000000ll - m.rbase;
    if (hi > 0) {
        m.tk_n = (uint32_t)hi;
        m.rb = (int32_t)(uint32_t)(uint64_t)m.rbase;
    }
}

// Workspace row of column c (top-k entry l_in for c >= W; -1 past the top-k
// columns), or -1.
__device__ __forceinline__ int ws_col(const WorkspaceIndexParams& p, const WsMeta& m, int c,
                                      int l_in) {
    if (c < p.window)
        return (uint32_t)(c - m.wc_lo) < m.wc_n ? (int)((uint32_t)m.wb + (uint32_t)c) : -1;
    return (uint32_t)l_in < m.tk_n ? (int)((uint32_t)m.rb + (uint32_t)l_in) : -1;
}

template <bool VEC, bool TMA>
__global__ void __launch_bounds__(kThreads) workspace_index_kernel(WorkspaceIndexParams p,
                                                                   int tokens_per_cta, int wpt) {
    extern __shared__ __align__(16) int32_t s_dyn[];  // TMA: the CTA's top-k rows
    __shared__ int s_cnt[kWarps];
    __shared__ __align__(8) uint64_t s_bar;
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t t0 = (int64_t)blockIdx.x * tokens_per_cta;
    int64_t t1 = t0 + tokens_per_cta;
    if (t1 > p.num_tokens) t1 = p.num_tokens;
    const int tpp = kWarps / wpt, tslot = warp / wpt, slice = warp % wpt;
    const int first = slice * kWarp + lane, stride = wpt * kWarp;
    const int W = p.window;
    const int P = (p.topk + 3) / 4 * 4;
    const int cols = W + P;
    const bool copy_topk = TMA && p.topk > 0;
    if (TMA && threadIdx.x == 0) {
        mbar_init(&s_bar, 1);
        mbar_fence_init();
    }
    if (TMA) __syncthreads();
    pdl_wait();
    pdl_launch_dependents();
    if (copy_topk && threadIdx.x == 0)
        stage_topk_rows(s_dyn, p.topk_local, p.topk_stride, p.topk, t0, t1, &s_bar);
    bool rows_ok = true;
    for (int64_t tb = t0; tb < t1; tb += tpp) {
        const int64_t t = tb + tslot;
        const int32_t* tk = p.topk_local + t * p.topk_stride;
        // The first batch of top-k quads depends only on t: issue it first.
        constexpr int kPre = PSK_WS_INDEX_BATCH;
        int4 Lpre[kPre];
        WsMeta m;
        m.ok = false;
        m.pos = m.lo = m.g0 = m.lc = m.rbase = 0;
        m.wc_lo = m.wb = m.rb = 0;
        m.wc_n = m.tk_n = 0u;
        if (t < t1) {
            const int32_t r = __ldg(p.t2r + t);
            if (VEC && !TMA) {
#pragma unroll
                for (int u = 0; u < kPre; ++u) {
                    const int q = first + u * stride;
                    const int c0 = 4 * q;
                    Lpre[u] = make_int4(-1, -1, -1, -1);
                    if (q < cols / 4 && c0 >= W) {
                        const int j0 = c0 - W;
                        if (j0 + 3 < p.topk) {
                            Lpre[u] = __ldg(reinterpret_cast<const int4*>(tk + j0));
                        } else {
                            Lpre[u].x = j0 < p.topk ? __ldg(tk + j0) : -1;
                            Lpre[u].y = j0 + 1 < p.topk ? __ldg(tk + j0 + 1) : -1;
                            Lpre[u].z = j0 + 2 < p.topk ? __ldg(tk + j0 + 2) : -1;
                        }
                    }
                }
            }
            m.ok = (p.valid == nullptr || __ldg(p.valid + t) != 0) && r >= 0 && r < p.num_reqs;
            if (m.ok) {
                const int64_t seq = __ldg(p.seq_lens + r);
                if (p.positions) {
                    m.pos = __ldg(p.positions + t);
                } else {
                    const int64_t qs = __ldg(p.qsl + r), qe = __ldg(p.qsl + r + 1);
                    m.pos = seq - (qe - qs) + (t - qs);
                }
                m.g0 = seq - __ldg(p.gather_lens + r);
                m.lc = seq / p.compress_ratio;
                m.rbase = (int64_t)r * p.workspace_width;
                m.lo = m.pos - W + 1;
                if (m.lo < 0) m.lo = 0;
            }
            ws_forms(p, m);
        }
        if (copy_topk && tb == t0) {
            rows_ok = mbar_wait_bounded(&s_bar, 0, kWaitLimitNs);
            if (!rows_ok && lane == 0) atomicAdd(&g_index_wait_timeouts, 1u);
        }
        int cnt = 0;
        if (t < t1 && rows_ok) {
            int32_t* out = p.out + t * p.out_stride;
            if (TMA) {
                const int32_t* s_row = s_dyn + (t - t0) * p.topk;
                const int nq = cols / 4;
#pragma unroll 2
                for (int q = first; q < nq; q += stride) {
                    const int c0 = 4 * q;
                    const int j0 = c0 - W;
                    const int4 l = (j0 >= 0 && j0 < p.topk)
                                       ? *reinterpret_cast<const int4*>(s_row + j0)
                                       : make_int4(-1, -1, -1, -1);
                    const int4 v = make_int4(ws_col(p, m, c0, l.x), ws_col(p, m, c0 + 1, l.y),
                                             ws_col(p, m, c0 + 2, l.z), ws_col(p, m, c0 + 3, l.w));
                    cnt += (v.x >= 0) + (v.y >= 0) + (v.z >= 0) + (v.w >= 0);
                    *reinterpret_cast<int4*>(out + c0) = v;
                }
            } else if (VEC) {
                constexpr int kBatch = PSK_WS_INDEX_BATCH;
                const int nq = cols / 4;
                for (int qb = first; qb < nq; qb += kBatch * stride) {
                    int4 L[kBatch];
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        const int q = qb + u * stride;
                        const int c0 = 4 * q;
                        L[u] = make_int4(-1, -1, -1, -1);
                        if (qb == first) {
                            L[u] = Lpre[u];
                        } else if (q < nq && c0 >= W) {
                            const int j0 = c0 - W;
                            if (j0 + 3 < p.topk) {
                                L[u] = __ldg(reinterpret_cast<const int4*>(tk + j0));
                            } else {
                                L[u].x = j0 < p.topk ? __ldg(tk + j0) : -1;
                                L[u].y = j0 + 1 < p.topk ? __ldg(tk + j0 + 1) : -1;
                                L[u].z = j0 + 2 < p.topk ? __ldg(tk + j0 + 2) : -1;
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        const int q = qb + u * stride;
                        if (q >= nq) break;
                        const int c0 = 4 * q;
                        const int4 l = L[u];
                        const int4 v = make_int4(ws_col(p, m, c0, l.x), ws_col(p, m, c0 + 1, l.y),
                                                 ws_col(p, m, c0 + 2, l.z), ws_col(p, m, c0 + 3, l.w));
                        cnt += (v.x >= 0) + (v.y >= 0) + (v.z >= 0) + (v.w >= 0);
                        *reinterpret_cast<int4*>(out + c0) = v;
                    }
                }
            } else {
                for (int c = first; c < cols; c += stride) {
                    const int l = (m.ok && c >= W && c - W < p.topk) ? __ldg(tk + (c - W)) : -1;
                    const int v = ws_col(p, m, c, l);
                    cnt += v >= 0;
                    out[c] = v;
                }
            }
        }
        cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
        if (wpt == 1) {
            if (lane == 0 && t < t1 && rows_ok) p.lens[t] = cnt;
        } else {
            if (lane == 0) s_cnt[warp] = cnt;
            __syncthreads();
            if (slice == 0 && lane == 0 && t < t1 && rows_ok) {
                int sum = 0;
                for (int i = 0; i < wpt; ++i) sum += s_cnt[warp + i];
                p.lens[t] = sum;
            }
            __syncthreads();
        }
    }
    if (copy_topk && !rows_ok && threadIdx.x == 0) mbar_wait_bounded(&s_bar, 0, kWaitLimitNs);
}

// ---- dense builders -------------------------------------------------------------------
//
// HCA decode (TokenSpeed backends/deepseek_v4.py,
// _decode_compressed_attention_indices_and_lens for a ratio other than 4) and
// the HCA prefill workspace's request-local form
// (_dense_prefill_local_compressed_indices): token t sees
// n = clamp(floor((pos + 1) / ratio), 0, width) compressed entries.  Every
// entry is arithmetic on the position, so one thread owns one 16-byte quad of
// one row (VEC) or one column; lens (= n, the global form) is written by the
// row's first thread.  No reduction, no shared memory.

// floor((pos + 1) / ratio) clamped to [0, width].
__device__ __forceinline__ int32_t visible_entries(int64_t pos, int32_t ratio, int32_t width) {
    const int64_t num = pos + 1;
    if (num <= 0) return 0;
    const int64_t n = num <= 0xFFFFFFFFll ? (int64_t)((uint32_t)num / (uint32_t)ratio)
                                          : num / ratio;
    return n < width ? (int32_t)n : width;
}

template <bool GLOBAL, bool VEC, bool POW2>
__global__ void __launch_bounds__(kThreads) dense_index_kernel(DenseParams p, TableRow tr0) {
    // at least one thread per row: it writes lens even when width is 0
    const int per_row = max(VEC ? (p.width + 3) / 4 : p.width, 1);
    const int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t t = g <= 0xFFFFFFFFll ? (int64_t)((uint32_t)g / (uint32_t)per_row) : g / per_row;
    const int q = (int)(g - t * per_row);
    pdl_wait();
    pdl_launch_dependents();
    if (t >= p.num_tokens) return;
    int32_t* out = p.out + t * p.out_stride;
    const int c0 = VEC ? 4 * q : q;
    constexpr int E = VEC ? 4 : 1;
    int v[4] = {-1, -1, -1, -1};
    if (GLOBAL) {
        const int32_t r = __ldg(p.t2r + t);
        const bool ok = (p.valid == nullptr || __ldg(p.valid + t) != 0) && r >= 0 &&
                        r < p.num_reqs;
        int32_t n = 0;
        if (ok) {
            n = visible_entries(__ldg(p.positions + t), p.ratio, p.width);
            TableRow tr = tr0;
            tr.row = p.bt + (int64_t)r * p.bt_stride;
            tr.base = p.base ? __ldg(p.base + r) : 0;
#pragma unroll
            for (int e = 0; e < E; ++e)
                if (c0 + e < n) v[e] = map_slot<false, POW2>(tr, c0 + e);
        }
        if (q == 0) p.lens[t] = n;
    } else {
        const int32_t n = visible_entries(__ldg(p.positions + t), p.ratio, p.width);
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (c0 + e < n) v[e] = c0 + e;
    }
    if (VEC && c0 + 3 < p.width) {
        *reinterpret_cast<int4*>(out + c0) = make_int4(v[0], v[1], v[2], v[3]);
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (c0 + e < p.width) out[c0 + e] = v[e];
    }
}

// Raises a kernel's dynamic shared-memory limit when a launch needs more than
// the default 48 KB (once per kernel and size class).
template <typename Kern>
cudaError_t allow_dynamic_smem(Kern kern, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t read_index_wait_timeouts(uint32_t* count) {
    return cudaMemcpyFromSymbol(count, g_index_wait_timeouts, sizeof(uint32_t));
}

cudaError_t launch_dense_indices(const DenseParams& p, bool global, cudaStream_t stream) {
    const bool vec = ((reinterpret_cast<uintptr_t>(p.out) & 15) == 0) && (p.out_stride % 4 == 0);
    const int64_t per_row = std::max<int64_t>(vec ? (p.width + 3) / 4 : p.width, 1);
    const int64_t threads = p.num_tokens * per_row;
    const int64_t blocks = (threads + kThreads - 1) / kThreads;
    TableRow tr{};
    tr.width = p.bt_width;
    tr.bs = p.bs;
    tr.shift = log2_if_pow2(p.bs);
    tr.maxp = INT_MAX / p.bs;
    tr.maxrem = INT_MAX % p.bs;
    const bool pow2 = tr.shift >= 0;
    using Kern = void (*)(DenseParams, TableRow);
    // [global][vec][pow2]
    static const Kern kTable[2][2][2] = {
        {{dense_index_kernel<false, false, false>, dense_index_kernel<false, false, true>},
         {dense_index_kernel<false, true, false>, dense_index_kernel<false, true, true>}},
        {{dense_index_kernel<true, false, false>, dense_index_kernel<true, false, true>},
         {dense_index_kernel<true, true, false>, dense_index_kernel<true, true, true>}}};
    return launch_pdl(kTable[global][vec][pow2], dim3((unsigned)blocks), dim3(kThreads), 0,
                      stream, p, tr);
}

cudaError_t launch_workspace_indices(const WorkspaceIndexParams& p, cudaStream_t stream) {
    const int sms = sm_count();
    const int64_t T = p.num_tokens;
    int wpt = 1;
    while (wpt < kWarps && T * wpt < (int64_t)sms * 16) wpt *= 2;
    const int tpp = kWarps / wpt;
    const bool vec = ((reinterpret_cast<uintptr_t>(p.out) & 15) == 0) && (p.out_stride % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(p.topk_local) & 15) == 0) &&
                     (p.topk_stride % 4 == 0) && (p.window % 4 == 0);
    // Staged top-k rows: one pass of tpp tokens per CTA, whole 16-byte quads.
    const bool tma = vec && p.topk % 4 == 0 && (int64_t)tpp * p.topk * 4 <= kMaxTopkStageBytes;
    int64_t passes = T / ((int64_t)tpp * 2 * sms);
    if (passes < 1) passes = 1;
    if (passes > PSK_WS_INDEX_MAX_PASSES) passes = PSK_WS_INDEX_MAX_PASSES;
    if (tma) passes = 1;
    const int tokens_per_cta = (int)(tpp * passes);
    const int64_t blocks = (T + tokens_per_cta - 1) / tokens_per_cta;
    const size_t smem = tma ? (size_t)tokens_per_cta * p.topk * sizeof(int32_t) : 0;
    auto kern = tma ? workspace_index_kernel<true, true>
                    : (vec ? workspace_index_kernel<true, false> : workspace_index_kernel<false, false>);
    const cudaError_t e = allow_dynamic_smem(kern, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), smem, stream, p, tokens_per_cta,
                      wpt);
}

cudaError_t launch_index_build(IndexParams p, bool has_swa, cudaStream_t stream) {
    const int sms = sm_count();
    const int64_t T = p.num_tokens;
    // Split a token over several warps when the batch is too small to fill
    // every SM with one warp per token.
    const int64_t want_warps = (int64_t)sms * PSK_INDEX_WARPS_PER_SM;
    int wpt = 1;
    while (wpt < kWarps && T * wpt < want_warps) wpt *= 2;
    const int tpp = kWarps / wpt;
    int64_t passes = T / ((int64_t)tpp * 2 * sms);
    if (passes < 1) passes = 1;
    if (passes > PSK_INDEX_MAX_PASSES) passes = PSK_INDEX_MAX_PASSES;
    p.warps_per_token = wpt;
    p.tokens_per_cta = (int32_t)(tpp * passes);
    p.stage_comp = (p.comp_width > 0 && p.comp_width <= kMaxStagedEntries) ? p.comp_width : 0;
    p.stage_swa = (has_swa && p.swa_width > 0 && p.swa_width <= kMaxStagedEntries) ? p.swa_width : 0;
    if (p.stage_comp == 0 || (has_swa && p.stage_swa == 0)) p.stage_comp = p.stage_swa = 0;
    const int64_t blocks = (T + p.tokens_per_cta - 1) / p.tokens_per_cta;
    p.comp_maxp = INT_MAX / p.comp_bs;
    p.comp_maxrem = INT_MAX % p.comp_bs;
    if (has_swa) {
        p.swa_maxp = INT_MAX / p.swa_bs;
        p.swa_maxrem = INT_MAX % p.swa_bs;
    }

    const bool vec = ((reinterpret_cast<uintptr_t>(p.out) & 15) == 0) && (p.out_stride % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(p.topk_local) & 15) == 0) &&
                     (p.topk_stride % 4 == 0) && (!has_swa || p.window % 4 == 0);
    // Top-k rows staged by bulk copies: whole 16-byte quads, at most
    // kMaxTopkStageBytes per CTA.
    const bool tma = vec && p.topk % 4 == 0 && p.tokens_per_cta <= kTopkBars &&
                     (int64_t)p.tokens_per_cta * p.topk * 4 <= kMaxTopkStageBytes;
    const bool pow2 = p.comp_shift >= 0 && (!has_swa || p.swa_shift >= 0);
    const size_t smem =
        ((tma ? (size_t)p.tokens_per_cta * p.topk : 0) + p.stage_comp + 1 + p.stage_swa + 1) *
        sizeof(int32_t);
    using Kern = void (*)(IndexParams);
    // [has_swa][pow2][mode: 0 scalar, 1 vector, 2 vector + staged top-k rows]
    static const Kern kTable[2][2][3] = {
        {{index_build_kernel<false, false, false, false>, index_build_kernel<false, true, false, false>,
          index_build_kernel<false, true, false, true>},
         {index_build_kernel<false, false, true, false>, index_build_kernel<false, true, true, false>,
          index_build_kernel<false, true, true, true>}},
        {{index_build_kernel<true, false, false, false>, index_build_kernel<true, true, false, false>,
          index_build_kernel<true, true, false, true>},
         {index_build_kernel<true, false, true, false>, index_build_kernel<true, true, true, false>,
          index_build_kernel<true, true, true, true>}}};
    Kern kern = kTable[has_swa][pow2][tma ? 2 : (vec ? 1 : 0)];
    if (tma && !has_swa && blocks > (int64_t)sms * PSK_INDEX_TMA_MIN_CTAS)
        kern = pow2 ? index_build_kernel<false, true, true, true, PSK_INDEX_TMA_MIN_CTAS_WIDE>
                    : index_build_kernel<false, true, false, true, PSK_INDEX_TMA_MIN_CTAS_WIDE>;
    const cudaError_t e = allow_dynamic_smem(kern, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), smem, stream, p);
}

}  // namespace psk
