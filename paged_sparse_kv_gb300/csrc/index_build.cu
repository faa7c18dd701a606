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
//  * The compressed block-table row of a CTA whose tokens all belong to one
//    request is staged in shared memory once, so the random top-k look-ups
//    hit shared memory instead of L1/L2 (the shared-memory block-table tile).
//  * lens is a warp reduction (__reduce_add_sync) of per-lane valid counts,
//    combined across the warps of a token in shared memory when a token is
//    split over several warps (small batches: every SM gets work).
#include <climits>

#include "launch.h"
#include "psk_common.cuh"

namespace psk {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / kWarp;
constexpr int kMaxStagedEntries = 8192;  // 32 KB of int32 page ids

struct TableRow {
    const int32_t* row;  // global row, or shared copy
    int32_t width;
    int64_t base;
    int32_t bs;
    int32_t shift;  // log2(bs) or -1
};

// Slot of logical position p (p >= 0) through one block-table row, or -1.
__device__ __forceinline__ int32_t map_slot(const TableRow& tr, bool shared, int64_t p) {
    int64_t q, rem;
    if (tr.shift >= 0) {
        q = p >> tr.shift;
        rem = p & ((1 << tr.shift) - 1);
    } else {
        q = p / tr.bs;
        rem = p - q * tr.bs;
    }
    const int64_t lp = q - tr.base;
    if (lp < 0 || lp >= tr.width) return -1;
    const int32_t page = shared ? tr.row[lp] : __ldg(tr.row + lp);
    if (page < 0) return -1;
    const int64_t s = (int64_t)page * tr.bs + rem;
    return s > INT_MAX ? -1 : (int32_t)s;
}

// Returns this lane's count of valid entries for token t.
template <bool HAS_SWA, bool VEC>
__device__ __forceinline__ int build_row(const IndexParams& p, int64_t t, int slice, int lane,
                                         int32_t staged_req, const int32_t* s_comp) {
    const int stride = p.warps_per_token * kWarp;
    const int first = slice * kWarp + lane;
    int32_t* out = p.out + t * p.out_stride;
    const int32_t r = __ldg(p.t2r + t);
    const bool ok = (p.valid == nullptr || __ldg(p.valid + t) != 0) && r >= 0 && r < p.num_reqs;
    if (!ok) {
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

    const bool use_s = (r == staged_req);
    TableRow comp;
    comp.row = use_s ? s_comp : p.comp_bt + (int64_t)r * p.comp_stride;
    comp.width = p.comp_width;
    comp.base = p.comp_base ? __ldg(p.comp_base + r) : 0;
    comp.bs = p.comp_bs;
    comp.shift = p.comp_shift;

    TableRow swa;
    int64_t pos = 0, lo = 0;
    if (HAS_SWA) {
        swa.row = p.swa_bt + (int64_t)r * p.swa_stride;
        swa.width = p.swa_width;
        swa.base = p.swa_base ? __ldg(p.swa_base + r) : 0;
        swa.bs = p.swa_bs;
        swa.shift = p.swa_shift;
        const int64_t qs = __ldg(p.qsl + r);
        const int64_t qe = __ldg(p.qsl + r + 1);
        pos = (int64_t)__ldg(p.seq_lens + r) - (qe - qs) + (t - qs);
        lo = pos - p.window + 1;
        const int64_t rs = p.replay ? (int64_t)__ldg(p.replay + r) : 0;
        if (rs > lo) lo = rs;
        if (lo < 0) lo = 0;
    }
    const int32_t* tk = p.topk_local + t * p.topk_stride;
    const int W = HAS_SWA ? p.window : 0;

    int cnt = 0;
    if (VEC) {
        const int nq = (p.out_cols + 3) / 4;
        for (int q = first; q < nq; q += stride) {
            const int c0 = 4 * q;
            int v[4];
            if (HAS_SWA && c0 < W) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int64_t ps = lo + c0 + e;
                    v[e] = ps <= pos ? map_slot(swa, false, ps) : -1;
                }
            } else {
                const int j0 = c0 - W;
                int l[4];
                if (j0 + 3 < p.topk) {
                    const int4 w = __ldg(reinterpret_cast<const int4*>(tk + j0));
                    l[0] = w.x; l[1] = w.y; l[2] = w.z; l[3] = w.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) l[e] = (j0 + e < p.topk) ? __ldg(tk + j0 + e) : -1;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = l[e] >= 0 ? map_slot(comp, use_s, l[e]) : -1;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) cnt += v[e] >= 0;
            if (c0 + 3 < p.out_cols) {
                *reinterpret_cast<int4*>(out + c0) = make_int4(v[0], v[1], v[2], v[3]);
            } else {
                for (int e = 0; c0 + e < p.out_cols; ++e) out[c0 + e] = v[e];
            }
        }
    } else {
        for (int c = first; c < p.out_cols; c += stride) {
            int v;
            if (HAS_SWA && c < W) {
                const int64_t ps = lo + c;
                v = ps <= pos ? map_slot(swa, false, ps) : -1;
            } else {
                const int j = c - W;
                const int l = j < p.topk ? __ldg(tk + j) : -1;
                v = l >= 0 ? map_slot(comp, use_s, l) : -1;
            }
            cnt += v >= 0;
            out[c] = v;
        }
    }
    return cnt;
}

template <bool HAS_SWA, bool VEC>
__global__ void __launch_bounds__(kThreads) index_build_kernel(IndexParams p) {
    extern __shared__ int32_t s_comp[];
    __shared__ int s_cnt[kWarps];
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t t0 = (int64_t)blockIdx.x * p.tokens_per_cta;
    int64_t t1 = t0 + p.tokens_per_cta;
    if (t1 > p.num_tokens) t1 = p.num_tokens;
    pdl_wait();
    pdl_launch_dependents();

    // Stage the compressed block-table row when the tile is one request.
    int32_t staged = -1;
    if (p.stage_comp > 0) {
        const int32_t r0 = __ldg(p.t2r + t0);
        const int32_t r1 = __ldg(p.t2r + t1 - 1);
        if (r0 == r1 && r0 >= 0 && r0 < p.num_reqs) staged = r0;
        if (staged >= 0) {
            const int32_t* src = p.comp_bt + (int64_t)staged * p.comp_stride;
            for (int i = threadIdx.x; i < p.stage_comp; i += kThreads) s_comp[i] = __ldg(src + i);
        }
        __syncthreads();
    }

    const int wpt = p.warps_per_token;
    const int tpp = kWarps / wpt;  // tokens per pass
    const int tslot = warp / wpt;
    const int slice = warp % wpt;
    for (int64_t tb = t0; tb < t1; tb += tpp) {
        const int64_t t = tb + tslot;
        int cnt = 0;
        if (t < t1) cnt = build_row<HAS_SWA, VEC>(p, t, slice, lane, staged, s_comp);
        cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
        if (wpt == 1) {
            if (lane == 0 && t < t1) p.lens[t] = cnt;
        } else {
            if (lane == 0) s_cnt[warp] = cnt;
            __syncthreads();
            if (slice == 0 && lane == 0 && t < t1) {
                int sum = 0;
                for (int i = 0; i < wpt; ++i) sum += s_cnt[warp + i];
                p.lens[t] = sum;
            }
            __syncthreads();
        }
    }
}

}  // namespace

cudaError_t launch_index_build(IndexParams p, bool has_swa, cudaStream_t stream) {
    const int sms = sm_count();
    const int64_t T = p.num_tokens;
    // Split a token over several warps when the batch is too small to fill
    // every SM with one warp per token.
    const int64_t want_warps = (int64_t)sms * 16;
    int wpt = 1;
    while (wpt < kWarps && T * wpt < want_warps) wpt *= 2;
    const int tpp = kWarps / wpt;
    int64_t passes = T / ((int64_t)tpp * 2 * sms);
    if (passes < 1) passes = 1;
    if (passes > 8) passes = 8;
    p.warps_per_token = wpt;
    p.tokens_per_cta = (int32_t)(tpp * passes);
    p.stage_comp = (p.comp_width > 0 && p.comp_width <= kMaxStagedEntries) ? p.comp_width : 0;
    const int64_t blocks = (T + p.tokens_per_cta - 1) / p.tokens_per_cta;
    const size_t smem = (size_t)p.stage_comp * sizeof(int32_t);

    const bool vec = ((reinterpret_cast<uintptr_t>(p.out) & 15) == 0) && (p.out_stride % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(p.topk_local) & 15) == 0) &&
                     (p.topk_stride % 4 == 0) && (!has_swa || p.window % 4 == 0);
    auto kern = has_swa ? (vec ? index_build_kernel<true, true> : index_build_kernel<true, false>)
                        : (vec ? index_build_kernel<false, true> : index_build_kernel<false, false>);
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), smem, stream, p);
}

}  // namespace psk
