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
#include <climits>

#include "launch.h"
#include "psk_common.cuh"

namespace psk {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / kWarp;
constexpr int kMaxStagedEntries = 4096;  // 16 KB of int32 page ids per staged row

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

// Per-token values that depend on its request (second memory round trip).
struct TokMeta {
    int32_t r;
    bool ok;
    int64_t pos, lo;
    int64_t swa_base, comp_base;
};

template <bool HAS_SWA>
__device__ __forceinline__ TokMeta load_meta(const IndexParams& p, int64_t t, int32_t r) {
    TokMeta m;
    m.r = r;
    m.ok = (p.valid == nullptr || __ldg(p.valid + t) != 0) && r >= 0 && r < p.num_reqs;
    m.pos = m.lo = 0;
    m.swa_base = m.comp_base = 0;
    if (!m.ok) return m;
    m.comp_base = p.comp_base ? __ldg(p.comp_base + r) : 0;
    if (HAS_SWA) {
        m.swa_base = p.swa_base ? __ldg(p.swa_base + r) : 0;
        const int64_t qs = __ldg(p.qsl + r);
        const int64_t qe = __ldg(p.qsl + r + 1);
        m.pos = (int64_t)__ldg(p.seq_lens + r) - (qe - qs) + (t - qs);
        int64_t lo = m.pos - p.window + 1;
        const int64_t rs = p.replay ? (int64_t)__ldg(p.replay + r) : 0;
        if (rs > lo) lo = rs;
        if (lo < 0) lo = 0;
        m.lo = lo;
    }
    return m;
}

// Loads the top-k quad that starts at output column c0 (-1 past topk).
__device__ __forceinline__ int4 load_topk_quad(const IndexParams& p, const int32_t* tk, int j0) {
    if (j0 + 3 < p.topk) return __ldg(reinterpret_cast<const int4*>(tk + j0));
    return make_int4(j0 < p.topk ? __ldg(tk + j0) : -1, j0 + 1 < p.topk ? __ldg(tk + j0 + 1) : -1,
                     j0 + 2 < p.topk ? __ldg(tk + j0 + 2) : -1, -1);
}

// Writes token t's row and returns this lane's count of valid entries.
// `pre` is the top-k quad of column group `first`, loaded in advance (VEC).
template <bool HAS_SWA, bool VEC>
__device__ __forceinline__ int build_row(const IndexParams& p, int64_t t, const TokMeta& m,
                                         int first, int stride, int4 pre, bool swa_s,
                                         bool comp_s, const int32_t* s_swa,
                                         const int32_t* s_comp) {
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
    comp.row = comp_s ? s_comp : p.comp_bt + (int64_t)m.r * p.comp_stride;
    comp.width = p.comp_width;
    comp.base = m.comp_base;
    comp.bs = p.comp_bs;
    comp.shift = p.comp_shift;
    TableRow swa;
    if (HAS_SWA) {
        swa.row = swa_s ? s_swa : p.swa_bt + (int64_t)m.r * p.swa_stride;
        swa.width = p.swa_width;
        swa.base = m.swa_base;
        swa.bs = p.swa_bs;
        swa.shift = p.swa_shift;
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
                    const int64_t ps = m.lo + c0 + e;
                    v[e] = ps <= m.pos ? map_slot(swa, swa_s, ps) : -1;
                }
            } else {
                const int4 w = (q == first) ? pre : load_topk_quad(p, tk, c0 - W);
                v[0] = w.x >= 0 ? map_slot(comp, comp_s, w.x) : -1;
                v[1] = w.y >= 0 ? map_slot(comp, comp_s, w.y) : -1;
                v[2] = w.z >= 0 ? map_slot(comp, comp_s, w.z) : -1;
                v[3] = w.w >= 0 ? map_slot(comp, comp_s, w.w) : -1;
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
    } else {
        for (int c = first; c < p.out_cols; c += stride) {
            int v;
            if (HAS_SWA && c < W) {
                const int64_t ps = m.lo + c;
                v = ps <= m.pos ? map_slot(swa, swa_s, ps) : -1;
            } else {
                const int j = c - W;
                const int l = j < p.topk ? __ldg(tk + j) : -1;
                v = l >= 0 ? map_slot(comp, comp_s, l) : -1;
            }
            cnt += v >= 0;
            out[c] = v;
        }
    }
    return cnt;
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

template <bool HAS_SWA, bool VEC>
__global__ void __launch_bounds__(kThreads) index_build_kernel(IndexParams p) {
    extern __shared__ int32_t s_tab[];  // [stage_comp] compressed row, then [stage_swa] SWA row
    __shared__ int s_cnt[kWarps];
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
    pdl_wait();
    pdl_launch_dependents();

    // Round 1: loads that depend only on token indices.
    const int32_t r0 = __ldg(p.t2r + t0);
    const int32_t r1 = __ldg(p.t2r + t1 - 1);
    const int64_t tf = t0 + tslot;  // this warp's first token
    int32_t rf = -1;
    int4 pre = make_int4(-1, -1, -1, -1);
    if (tf < t1) {
        rf = __ldg(p.t2r + tf);
        if (VEC && 4 * first >= W && 4 * first < p.out_cols)
            pre = load_topk_quad(p, p.topk_local + tf * p.topk_stride, 4 * first - W);
    }
    // Round 2: the first token's request metadata and, when the tile is one
    // request, its block-table rows into shared memory.
    TokMeta mf;
    if (tf < t1) mf = load_meta<HAS_SWA>(p, tf, rf);
    const int32_t staged = (r0 == r1 && r0 >= 0 && r0 < p.num_reqs) ? r0 : -1;
    const bool comp_s = staged >= 0 && p.stage_comp > 0;
    const bool swa_s = HAS_SWA && staged >= 0 && p.stage_swa > 0;
    int32_t* s_comp = s_tab;
    int32_t* s_swa = s_tab + p.stage_comp;
    if (comp_s) stage_row(s_comp, p.comp_bt + (int64_t)staged * p.comp_stride, p.stage_comp);
    if (swa_s) stage_row(s_swa, p.swa_bt + (int64_t)staged * p.swa_stride, p.stage_swa);
    __syncthreads();

    for (int64_t tb = t0; tb < t1; tb += tpp) {
        const int64_t t = tb + tslot;
        int cnt = 0;
        if (t < t1) {
            TokMeta m;
            int4 q0;
            if (tb == t0) {
                m = mf;
                q0 = pre;
            } else {
                m = load_meta<HAS_SWA>(p, t, __ldg(p.t2r + t));
                q0 = (VEC && 4 * first >= W && 4 * first < p.out_cols)
                         ? load_topk_quad(p, p.topk_local + t * p.topk_stride, 4 * first - W)
                         : make_int4(-1, -1, -1, -1);
            }
            const bool same = m.r == staged;
            cnt = build_row<HAS_SWA, VEC>(p, t, m, first, stride, q0, swa_s && same,
                                          comp_s && same, s_swa, s_comp);
        }
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

// ---- workspace-relative form ------------------------------------------------------
//
// TokenSpeed's combine_topk_swa_indices as the prefill workspace path calls it
// (backends/deepseek_v4.py, _prefill_workspace): request r's rows start at
// r * workspace_width, compressed entries at rows 0.., the gathered window
// positions g0 = seq - gather_len .. seq - 1 at rows compressed_base...  No
// table look-ups: every column is arithmetic on the token's metadata.
template <bool VEC>
__global__ void __launch_bounds__(kThreads) workspace_index_kernel(WorkspaceIndexParams p,
                                                                   int tokens_per_cta, int wpt) {
    __shared__ int s_cnt[kWarps];
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int64_t t0 = (int64_t)blockIdx.x * tokens_per_cta;
    int64_t t1 = t0 + tokens_per_cta;
    if (t1 > p.num_tokens) t1 = p.num_tokens;
    const int tpp = kWarps / wpt, tslot = warp / wpt, slice = warp % wpt;
    const int first = slice * kWarp + lane, stride = wpt * kWarp;
    const int W = p.window;
    const int P = (p.topk + 3) / 4 * 4;
    const int cols = W + P;
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t tb = t0; tb < t1; tb += tpp) {
        const int64_t t = tb + tslot;
        int cnt = 0;
        if (t < t1) {
            int32_t* out = p.out + t * p.out_stride;
            const int32_t r = __ldg(p.t2r + t);
            const bool ok = (p.valid == nullptr || __ldg(p.valid + t) != 0) && r >= 0 &&
                            r < p.num_reqs;
            int64_t pos = 0, lo = 0, g0 = 0, lc = 0, rbase = 0;
            if (ok) {
                const int64_t qs = __ldg(p.qsl + r), qe = __ldg(p.qsl + r + 1);
                const int64_t seq = __ldg(p.seq_lens + r);
                pos = seq - (qe - qs) + (t - qs);
                g0 = seq - __ldg(p.gather_lens + r);
                lc = seq / p.compress_ratio;
                rbase = (int64_t)r * p.workspace_width;
                lo = pos - W + 1;
                if (lo < 0) lo = 0;
            }
            const int32_t* tk = p.topk_local + t * p.topk_stride;
            auto col = [&](int c, int l_in) -> int {
                if (!ok) return -1;
                int64_t v = -1;
                if (c < W) {
                    const int64_t ps = lo + c;
                    if (ps <= pos && ps >= g0) v = rbase + p.compressed_base + (ps - g0);
                } else if (c - W < p.topk) {
                    if (l_in >= 0 && l_in < lc) v = rbase + l_in;
                }
                return v > 0x7FFFFFFFll ? -1 : (int)v;
            };
            if (VEC) {
                const int nq = cols / 4;
                for (int q = first; q < nq; q += stride) {
                    const int c0 = 4 * q;
                    int4 l = make_int4(-1, -1, -1, -1);
                    if (ok && c0 >= W) {
                        const int j0 = c0 - W;
                        if (j0 + 3 < p.topk) {
                            l = __ldg(reinterpret_cast<const int4*>(tk + j0));
                        } else {
                            l.x = j0 < p.topk ? __ldg(tk + j0) : -1;
                            l.y = j0 + 1 < p.topk ? __ldg(tk + j0 + 1) : -1;
                            l.z = j0 + 2 < p.topk ? __ldg(tk + j0 + 2) : -1;
                        }
                    }
                    const int4 v = make_int4(col(c0, l.x), col(c0 + 1, l.y), col(c0 + 2, l.z),
                                             col(c0 + 3, l.w));
                    cnt += (v.x >= 0) + (v.y >= 0) + (v.z >= 0) + (v.w >= 0);
                    *reinterpret_cast<int4*>(out + c0) = v;
                }
            } else {
                for (int c = first; c < cols; c += stride) {
                    const int l = (ok && c >= W && c - W < p.topk) ? __ldg(tk + (c - W)) : -1;
                    const int v = col(c, l);
                    cnt += v >= 0;
                    out[c] = v;
                }
            }
        }
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

cudaError_t launch_workspace_indices(const WorkspaceIndexParams& p, cudaStream_t stream) {
    const int sms = sm_count();
    const int64_t T = p.num_tokens;
    int wpt = 1;
    while (wpt < kWarps && T * wpt < (int64_t)sms * 16) wpt *= 2;
    const int tpp = kWarps / wpt;
    int64_t passes = T / ((int64_t)tpp * 2 * sms);
    if (passes < 1) passes = 1;
    if (passes > 8) passes = 8;
    const int tokens_per_cta = (int)(tpp * passes);
    const int64_t blocks = (T + tokens_per_cta - 1) / tokens_per_cta;
    const bool vec = ((reinterpret_cast<uintptr_t>(p.out) & 15) == 0) && (p.out_stride % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(p.topk_local) & 15) == 0) &&
                     (p.topk_stride % 4 == 0) && (p.window % 4 == 0);
    auto kern = vec ? workspace_index_kernel<true> : workspace_index_kernel<false>;
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), 0, stream, p, tokens_per_cta,
                      wpt);
}

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
    p.stage_swa = (has_swa && p.swa_width > 0 && p.swa_width <= kMaxStagedEntries) ? p.swa_width : 0;
    const int64_t blocks = (T + p.tokens_per_cta - 1) / p.tokens_per_cta;
    const size_t smem = (size_t)(p.stage_comp + p.stage_swa) * sizeof(int32_t);

    const bool vec = ((reinterpret_cast<uintptr_t>(p.out) & 15) == 0) && (p.out_stride % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(p.topk_local) & 15) == 0) &&
                     (p.topk_stride % 4 == 0) && (!has_swa || p.window % 4 == 0);
    auto kern = has_swa ? (vec ? index_build_kernel<true, true> : index_build_kernel<true, false>)
                        : (vec ? index_build_kernel<false, true> : index_build_kernel<false, false>);
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), smem, stream, p);
}

}  // namespace psk
