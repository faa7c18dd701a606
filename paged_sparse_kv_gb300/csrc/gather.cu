// gather.cu -- index-keyed dequantize-and-gather.
//
// Per-row math: TokenSpeed deepseek_v4_ops.py,
// dequantize_deepseek_v4_fp8_ds_mla_cache (fp8_ds_mla) and
// read_deepseek_v4_indexer_mxfp4_cache (MXFP4); index form of vLLM
// deepseek_v41 ops dequantize_and_gather_k_cache.
//
// Two kernels:
//  * fp8_ds_mla records (584 B per 512-dim row): a warp-specialised pipeline
//    that moves records into shared memory with 1-D bulk copies (TMA) and
//    dequantizes from there (details above the kernel).
//  * MXFP4 records (68 B per 128-dim row): batched plain loads.
// Both write each output row as 32-byte chunks (one 256-bit store per lane
// when the output is 32-byte aligned), a warp store instruction covering up to
// 1 KB of contiguous output, issued as streaming (evict-first) stores so the
// gathered output does not push reused cache rows out of L2.  Decode is
// exact: cvt.rn.f16x2.{e4m3x2,e2m1x2}, a binary32 multiply by the scale, and
// cvt.rn.bf16x2.f32.  Invalid slots (negative or beyond the cache) give zero
// rows.  The scale multiply is one packed mul.rn.f32x2 per pair of elements.
#include "gather.h"
#include "psk_common.cuh"

namespace psk {
namespace {

constexpr int kThreads = 256;

// ---- fp8_ds_mla: warp-specialised TMA pipeline ------------------------------------
//
// Warp 0 (producer) walks tiles of kRowsPerTile consecutive (t, j) items: its
// lanes load the tile's slot ids with one coalesced load, then each lane issues
// a 1-D bulk copy (cp.async.bulk) of its row's data record and of the 16-byte
// aligned chunk holding the row's scales into stage s of a kStages-deep
// shared-memory ring, completing on the stage's `full` mbarrier
// (expect_tx = bytes of the valid rows).  The kConsumerWarps consumer warps
// wait on `full`, dequantize rows out of shared memory, stream them to global
// memory, and release the stage on its `empty` mbarrier.  The producer runs up
// to kStages tiles ahead, so each SM keeps tens of KB of row reads in flight
// without spending registers on them.  Every wait is bounded (2 s): on expiry
// the thread counts a timeout in g_wait_timeouts and stops; the producer
// always drains the copies it issued before it exits.

// Ring depth and residency of the FP8 gather: three stages of 16 rows (29 KB of
// shared memory at head_dim 512) and launch bounds for six CTAs per SM up to
// head_dim 512, which hold the kernel to 32 registers, so seven are resident.
// Against four stages at five CTAs per SM (40 registers), interleaved on one
// box, each launch alone after an L2 flush: the prefill top-k gather 1585 ->
// 1475 us, its window gather 401 -> 383 us, the fused top-k and window forms
// 1661 -> 1449 / 498 -> 387 us, the mixed window gather 110.6 -> 106.5 us; the
// mixed top-k gather (many padding entries, whose zero rows need no record and
// let the consumers outrun a shallower ring) 779 -> 817 us.  Six and eight
// stages at fewer CTAs per SM were slower still; boxes differ by up to ~9% on
// the same build.
#ifndef PSK_GATHER_STAGES
#define PSK_GATHER_STAGES 3
#endif
#ifndef PSK_GATHER_MIN_CTAS
#define PSK_GATHER_MIN_CTAS 6
#endif
constexpr int kStages = PSK_GATHER_STAGES;
constexpr int kRowsPerTile = 16;
constexpr int kConsumerWarps = 8;
constexpr int kTmaThreads = kWarp * (1 + kConsumerWarps);
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ unsigned int g_wait_timeouts = 0;

// 1 when every output row start (out + a * stride_a + b * stride_b elements)
// is 32-byte aligned, so a gather can store 32-byte chunks.
inline int out32_aligned(const void* out, int64_t stride_a, int64_t stride_b) {
    return (reinterpret_cast<uintptr_t>(out) % 32 == 0 && (stride_a * 2) % 32 == 0 &&
            (stride_b * 2) % 32 == 0) ? 1 : 0;
}

// Shuffle of a 32- or 64-bit record offset from lane `src`.
__device__ __forceinline__ uint32_t shfl_off(uint32_t v, int src) {
    return __shfl_sync(0xFFFFFFFFu, v, src);
}
__device__ __forceinline__ uint64_t shfl_off(uint64_t v, int src) {
    return __shfl_sync(0xFFFFFFFFu, (unsigned long long)v, src);
}

__device__ __forceinline__ void item_to_tj(int64_t item, int32_t cols, bool small, int64_t& t,
                                           int32_t& j) {
    if (small) {
        const uint32_t ui = (uint32_t)item, uc = (uint32_t)cols;
        const uint32_t q = ui / uc;
        t = q;
        j = (int32_t)(ui - q * uc);
    } else {
        t = item / cols;
        j = (int32_t)(item - t * cols);
    }
}

// Where each item's slot comes from: the index matrix (INDEX form), a
// request's position range through its block-table row (RANGE form), a
// token's local top-k index through its request's table (TOPK form) or a
// token's window position through the SWA table (WINDOW form).
enum : int { kSrcIndex = 0, kSrcRange = 1, kSrcTopk = 2, kSrcWindow = 3, kSrcPair = 4,
              kSrcDense = 5 };

struct ItemSource {
    GatherParams g;      // index form (and cache geometry and output for every form)
    RangeParams r;       // range form
    TopkSource tk;       // top-k form
    WindowSource wn;     // window form
    PairSource pr;       // pair form: index form over two caches split by column
    DenseSource ds;      // dense form: every visible compressed entry of a token
};

// Slot of position p through one table row (the block-table rule), or -1.
__device__ __forceinline__ int32_t table_slot(const int32_t* row, int32_t width, int64_t base,
                                              int32_t bs, int32_t shift, int64_t p) {
    if (p < 0) return -1;
    int64_t rem;
    const int64_t q = div_block(p, bs, shift, rem);
    const int64_t lp = q - base;
    if (lp < 0 || lp >= width) return -1;
    const int32_t page = __ldg(row + lp);
    if (page < 0) return -1;
    const int64_t s = (int64_t)page * bs + rem;
    return s > 0x7FFFFFFFll ? -1 : (int32_t)s;
}

// Slot of item (t, j) of the TOPK form: the compute_global_topk_indices_and_lens
// rule (padding token or -1 entry -> -1) then the gather's capacity check.
// The token's request, validity and top-k entry are loaded together.
__device__ __forceinline__ int32_t topk_item_slot(const TopkSource& s, int32_t bs, int32_t shift,
                                                  int64_t capacity, int64_t t, int32_t j) {
    const int32_t r = __ldg(s.t2r + t);
    const bool valid = s.valid == nullptr || __ldg(s.valid + t) != 0;
    const int32_t l = __ldg(s.topk_local + t * s.topk_stride + j);
    if (!valid || r < 0 || r >= s.num_reqs || l < 0) return -1;
    const int64_t base = s.base ? __ldg(s.base + r) : 0;
    const int32_t raw = table_slot(s.bt + (int64_t)r * s.bt_stride, s.bt_width, base, bs, shift, l);
    return (raw >= 0 && (int64_t)raw < capacity) ? raw : -1;
}

// Slot of window column c of token t (the WINDOW form): the window rule of
// combine_topk_swa_indices -- position from the request's metadata, window
// [max(replay_start, pos - W + 1, 0), pos], left-aligned -- then the gather's
// capacity check.
__device__ __forceinline__ int32_t window_item_slot(const WindowSource& s, int32_t W, int32_t bs,
                                                    int32_t shift, int64_t capacity, int64_t t,
                                                    int32_t c) {
    const int32_t r = __ldg(s.t2r + t);
    const bool valid = s.valid == nullptr || __ldg(s.valid + t) != 0;
    if (!valid || r < 0 || r >= s.num_reqs) return -1;
    const int64_t qs = __ldg(s.qsl + r), qe = __ldg(s.qsl + r + 1);
    const int64_t seq = __ldg(s.seq_lens + r);
    const int64_t rs = s.replay ? (int64_t)__ldg(s.replay + r) : 0;
    const int64_t base = s.base ? __ldg(s.base + r) : 0;
    const int64_t pos = seq - (qe - qs) + (t - qs);
    int64_t lo = pos - W + 1;
    if (rs > lo) lo = rs;
    if (lo < 0) lo = 0;
    const int64_t p = lo + c;
    if (p > pos) return -1;
    const int32_t raw = table_slot(s.bt + (int64_t)r * s.bt_stride, s.bt_width, base, bs, shift, p);
    return (raw >= 0 && (int64_t)raw < capacity) ? raw : -1;
}

// Slot of item (t, c) of the DENSE form: the rule of
// compute_dense_compressed_indices_and_lens (padding token -> -1; entries past
// the visible count -> -1) then the gather's capacity check.
__device__ __forceinline__ int32_t dense_item_slot(const DenseSource& s, int32_t cols, int32_t bs,
                                                   int32_t shift, int64_t capacity, int64_t t,
                                                   int32_t c) {
    const int32_t r = __ldg(s.t2r + t);
    const bool valid = s.valid == nullptr || __ldg(s.valid + t) != 0;
    if (!valid || r < 0 || r >= s.num_reqs) return -1;
    const int64_t num = __ldg(s.positions + t) + 1;
    if (num <= 0) return -1;
    const int64_t n = num <= 0xFFFFFFFFll ? (int64_t)((uint32_t)num / (uint32_t)s.ratio)
                                          : num / s.ratio;
    if (c >= n || c >= cols) return -1;
    const int64_t base = s.base ? __ldg(s.base + r) : 0;
    const int32_t raw = table_slot(s.bt + (int64_t)r * s.bt_stride, s.bt_width, base, bs, shift, c);
    return (raw >= 0 && (int64_t)raw < capacity) ? raw : -1;
}

template <int D, bool UE8M0, int SRC>
__global__ void __launch_bounds__(kTmaThreads, D <= 512 ? PSK_GATHER_MIN_CTAS : 1)
gather_fp8_tma_kernel(ItemSource src, int slot_bytes, int v8) {
    const GatherParams& p = src.g;
    // A consumer lane owns 32-byte output chunks (16 bf16 values): with a
    // 32-byte aligned output each is one 256-bit store and a warp's store covers
    // 1 KB of contiguous output (v8 != 0), else two 16-byte stores.
    constexpr int CHUNKS = D / 16;
    constexpr int LANES = CHUNKS < kWarp ? CHUNKS : kWarp;
    constexpr int CPL = CHUNKS / LANES;
    constexpr int GPW = kWarp / LANES;
    constexpr int NBLK = D / 64;
    constexpr int SDIM = UE8M0 ? NBLK : 4 * NBLK;

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kRowsPerTile * slot_bytes);
    uint64_t* empty = full + kStages;
    int64_t* outoff = reinterpret_cast<int64_t*>(empty + kStages);   // [kStages][kRowsPerTile]
    int32_t* slots = reinterpret_cast<int32_t*>(outoff + kStages * kRowsPerTile);

    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    // INDEX form: items = rows x cols of the index matrix.  RANGE form:
    // items = num_reqs x span, span = out_rows - offset rows per request.
    constexpr bool RANGE = SRC == kSrcRange;
    const int64_t span = RANGE ? src.r.out_rows - src.r.offset : (int64_t)p.cols;
    const int64_t items = RANGE ? (int64_t)src.r.num_reqs * span : p.rows * (int64_t)p.cols;
    const int64_t tiles = (items + kRowsPerTile - 1) / kRowsPerTile;
    const int64_t capacity = p.num_pages * (int64_t)p.block_size;
    const int64_t capacity2 = SRC == kSrcPair ? src.pr.num_pages * (int64_t)src.pr.block_size : 0;
    const bool small = items <= 0xFFFFFFFFll && span <= 0x7FFFFFFFll;
    const int nope = D - p.rope_dim;
    const int ts = nope + 2 * p.rope_dim;
    const int bs = p.block_size;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_fence_init();
    }
    __syncthreads();
    // Every input, the slot metadata included, may come from the previous
    // kernel on the stream: nothing global is read before its grid is done.
    pdl_wait();
    pdl_launch_dependents();

    if (warp == 0) {
        // Producer.  Lanes 0-15 and 16-31 load the slot ids of two tiles per
        // load instruction; each round covers kLoadTiles tiles, so the ring
        // fills after one index-load latency instead of one per tile.
        constexpr int kLoadTiles = 4;
        const int half = lane >> 4, r = lane & 15;
        int i = 0;
        bool ok = true;
        for (int64_t base = blockIdx.x; base < tiles && ok; base += (int64_t)kLoadTiles * gridDim.x) {
            int32_t slot[kLoadTiles / 2];
            int64_t oof[kLoadTiles / 2];
            bool second[kLoadTiles / 2];  // PAIR form: the item reads the second cache
#pragma unroll
            for (int q = 0; q < kLoadTiles / 2; ++q) {
                const int64_t tile = base + (int64_t)(2 * q + half) * gridDim.x;
                const int64_t item = tile * kRowsPerTile + r;
                slot[q] = -1;
                oof[q] = 0;
                second[q] = false;
                if (tile < tiles && item < items) {
                    int64_t t;
                    int32_t j;
                    item_to_tj(item, (int32_t)span, small, t, j);
                    if (RANGE) {
                        // t = request, j = row within the request's span
                        const int64_t seq = __ldg(src.r.seq_lens + t);
                        const int64_t g = src.r.gather_lens ? __ldg(src.r.gather_lens + t) : seq;
                        if (j < g) {
                            const int64_t base = src.r.base_offsets ? __ldg(src.r.base_offsets + t) : 0;
                            const int32_t raw = table_slot(src.r.block_table + t * src.r.bt_stride,
                                                           src.r.bt_width, base, p.block_size,
                                                           p.block_shift, seq - g + j);
                            slot[q] = (raw >= 0 && (int64_t)raw < capacity) ? raw : -1;
                            oof[q] = t * src.r.out_stride_r + (src.r.offset + j) * src.r.out_stride_i;
                        } else {
                            slot[q] = -2;  // outside the gathered range: not written
                        }
                    } else {
                        if (SRC == kSrcTopk) {
                            slot[q] = topk_item_slot(src.tk, bs, p.block_shift, capacity, t, j);
                        } else if (SRC == kSrcWindow) {
                            slot[q] = window_item_slot(src.wn, p.cols, bs, p.block_shift, capacity,
                                                       t, j);
                        } else if (SRC == kSrcDense) {
                            slot[q] = dense_item_slot(src.ds, p.cols, bs, p.block_shift, capacity,
                                                      t, j);
                        } else if (SRC == kSrcPair) {
                            second[q] = j >= src.pr.split;
                            const int64_t cap = second[q] ? capacity2 : capacity;
                            const int32_t raw = __ldg(p.idx + t * p.idx_stride + j);
                            slot[q] = (raw >= 0 && (int64_t)raw < cap) ? raw : -1;
                        } else {
                            const int32_t raw = __ldg(p.idx + t * p.idx_stride + j);
                            slot[q] = (raw >= 0 && (int64_t)raw < capacity) ? raw : -1;
                        }
                        oof[q] = t * p.out_stride_t + (int64_t)j * p.out_stride_j;
                    }
                } else {
                    slot[q] = -2;
                }
            }
#pragma unroll
            for (int k = 0; k < kLoadTiles; ++k) {
                const int64_t tile = base + (int64_t)k * gridDim.x;
                if (tile >= tiles) break;
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait_bounded(&empty[s], ((i / kStages) - 1) & 1, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                const bool mine = half == (k & 1);
                const int32_t sl = mine ? slot[k / 2] : -2;
                uint32_t bytes = 0;
                const uint8_t* src_data = nullptr;
                const uint8_t* src_scl = nullptr;
                uint32_t scl_bytes = 0;
                int32_t soff = -1;
                if (sl >= 0) {
                    const bool sec = SRC == kSrcPair && mine && second[k / 2];
                    const int32_t cbs = sec ? src.pr.block_size : bs;
                    int32_t off;
                    const int32_t page = div_block32(sl, cbs, sec ? src.pr.block_shift : p.block_shift, off);
                    const uint8_t* pbase = (sec ? src.pr.cache : p.cache) +
                                           (int64_t)page * (sec ? src.pr.page_stride : p.page_stride);
                    src_data = pbase + (int64_t)off * ts;
                    const uintptr_t a = reinterpret_cast<uintptr_t>(pbase + (int64_t)cbs * ts + (int64_t)off * SDIM);
                    const uintptr_t a0 = a & ~(uintptr_t)15, a1 = (a + SDIM + 15) & ~(uintptr_t)15;
                    src_scl = reinterpret_cast<const uint8_t*>(a0);
                    scl_bytes = (uint32_t)(a1 - a0);
                    soff = (int32_t)(a - a0);
                    bytes = (uint32_t)ts + scl_bytes;
                }
                const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, bytes);
                if (mine) {
                    slots[s * kRowsPerTile + r] = sl == -2 ? -2 : soff;  // -1 zero row, -2 skip
                    outoff[s * kRowsPerTile + r] = oof[k / 2];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(&full[s], total);
                __syncwarp();
                if (sl >= 0) {
                    uint8_t* dst = ring + (size_t)(s * kRowsPerTile + r) * slot_bytes;
                    bulk_g2s(dst, src_data, (uint32_t)ts, &full[s]);
                    bulk_g2s(dst + ts, src_scl, scl_bytes, &full[s]);
                }
                ++i;
            }
        }
        if (!ok && lane == 0) atomicAdd(&g_wait_timeouts, 1u);
        // Drain: the last phase issued on every stage must land before exit.
        if (lane == 0) {
            for (int s = 0; s < kStages && s < i; ++s) {
                const int last = s + ((i - 1 - s) / kStages) * kStages;
                if (!mbar_wait_bounded(&full[s], (last / kStages) & 1, kWaitLimitNs))
                    atomicAdd(&g_wait_timeouts, 1u);
            }
        }
        return;
    }

    const int cw = warp - 1;
    const int grp = lane / LANES, gl = lane % LANES;
    int i = 0;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++i) {
        const int s = i % kStages;
        if (!mbar_wait_bounded(&full[s], (i / kStages) & 1, kWaitLimitNs)) {
            if (lane == 0) atomicAdd(&g_wait_timeouts, 1u);
            return;
        }
        for (int r = cw * GPW + grp; r < kRowsPerTile; r += kConsumerWarps * GPW) {
            const int64_t item = tile * kRowsPerTile + r;
            if (item >= items) break;
            const int32_t soff = slots[s * kRowsPerTile + r];  // scale offset, -1 = zero row
            if (soff == -2) continue;                           // not written
            uint16_t* orow = p.out + outoff[s * kRowsPerTile + r];
            const uint8_t* srow = ring + (size_t)(s * kRowsPerTile + r) * slot_bytes;
#pragma unroll
            for (int ci = 0; ci < CPL; ++ci) {
                const int c = gl + ci * LANES;  // values [16c, 16c + 16)
                uint4 lo, hi;
                if (soff < 0) {
                    lo = hi = make_uint4(0u, 0u, 0u, 0u);
                } else if (16 * c < nope) {
                    const uint4 w = lds_v4(srow + 16 * c);
                    float sc;
                    if constexpr (UE8M0) {
                        sc = ue8m0_scale(lds_u8(srow + ts + soff + c / 4));
                    } else {
                        sc = __uint_as_float(lds_u32(srow + ts + soff + 4 * (c / 4)));
                    }
                    const uint64_t s2 = splat_f32x2(sc);
                    lo.x = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.x & 0xFFFFu), s2);
                    lo.y = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.x >> 16), s2);
                    lo.z = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.y & 0xFFFFu), s2);
                    lo.w = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.y >> 16), s2);
                    hi.x = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.z & 0xFFFFu), s2);
                    hi.y = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.z >> 16), s2);
                    hi.z = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.w & 0xFFFFu), s2);
                    hi.w = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.w >> 16), s2);
                } else {
                    // RoPE values: bf16 bytes [nope + 2 (16c - nope), + 32) of the record
                    lo = lds_v4(srow + 32 * c - nope);
                    hi = lds_v4(srow + 32 * c - nope + 16);
                }
                store_out32(orow + 16 * c, lo, hi, v8);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// ---- small records (MXFP4, FP8 indexer): batched loads --------------------------------
//
// A 68-byte MXFP4 record (or a 132-byte FP8 indexer record at head_dim 128)
// is too small for a bulk copy to pay off, so this gather uses plain loads
// arranged for memory-level parallelism.  A warp resolves up to 32 consecutive
// (t, j) items at a time (rpr of them), one per lane: the item's slot (from the index
// matrix, or its local top-k entry through the request's table), the byte
// offsets of its record's values and scales in the cache, and its output
// offset.  It then walks those items in groups of STEPS * GPW: each lane group
// takes an item's offsets from the owner lane by shuffles, every record load
// of the group (per lane and item: 8 bytes of packed E2M1 values and their
// scale byte, or 16 e4m3 bytes and the row's binary32 scale) is issued before
// any conversion, then the group is converted and each lane stores its 16
// values as one 32-byte chunk.  Offsets are 32-bit
// when the cache is below 4 GiB (OFF = uint32_t), else 64-bit.
// REC 1: MXFP4 (TokenSpeed read_deepseek_v4_indexer_mxfp4_cache); REC 2: the
// FP8 indexer record (write_deepseek_v4_indexer_fp8_cache's layout).
// Rows per lane group in one group of the small-record gather.
constexpr int kSmallSteps = 4;

template <int D, int REC, int SRC, typename OFF>
__global__ void __launch_bounds__(kThreads)
gather_small_kernel(GatherParams p, TopkSource tk, int rpr, int v8) {
    constexpr int CHUNKS = D / 16;  // 32-byte output chunks (16 values) per row
    constexpr int LANES = CHUNKS < kWarp ? CHUNKS : kWarp;
    constexpr int CPL = CHUNKS / LANES;
    constexpr int GPW = kWarp / LANES;
    constexpr int STEPS = (kWarp / GPW) < kSmallSteps ? (kWarp / GPW) : kSmallSteps;
    constexpr int GROUP = STEPS * GPW;          // items per group, a divisor of 32
    constexpr int VB = REC == 1 ? D / 2 : D;    // value bytes per token
    constexpr int SB = REC == 1 ? D / 32 : 4;   // scale bytes per token
    constexpr OFF kZeroRow = ~(OFF)0;           // value offset of an item with no record

    const int lane = threadIdx.x & 31;
    const int grp = lane / LANES, gl = lane % LANES;
    const int64_t warp_id = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / kWarp;
    const int64_t nwarps = (int64_t)gridDim.x * kThreads / kWarp;
    const int64_t items = p.rows * (int64_t)p.cols;
    const int64_t capacity = p.num_pages * (int64_t)p.block_size;
    const bool small = items <= 0xFFFFFFFFll;
    const OFF scale_region = (OFF)((int64_t)p.block_size * VB);
    pdl_wait();
    pdl_launch_dependents();

    for (int64_t b0 = warp_id * rpr; b0 < items; b0 += nwarps * rpr) {
        // item b0 + lane (lane < rpr): its record's value and scale offsets and
        // its output offset
        OFF my_vo = kZeroRow, my_so = 0;
        int64_t my_out = -1;
        if (lane < rpr && b0 + lane < items) {
            const int64_t item = b0 + lane;
            int64_t t;
            int32_t j;
            if (small) {
                const uint32_t q = (uint32_t)item / (uint32_t)p.cols;
                t = q;
                j = (int32_t)((uint32_t)item - q * (uint32_t)p.cols);
            } else {
                t = item / p.cols;
                j = (int32_t)(item - t * p.cols);
            }
            int32_t slot;
            if (SRC == kSrcTopk) {
                slot = topk_item_slot(tk, p.block_size, p.block_shift, capacity, t, j);
            } else {
                const int32_t raw = __ldg(p.idx + t * p.idx_stride + j);
                slot = (raw >= 0 && (int64_t)raw < capacity) ? raw : -1;
            }
            if (slot >= 0) {
                int32_t off;
                const int32_t page = div_block32(slot, p.block_size, p.block_shift, off);
                const OFF pb = (OFF)((int64_t)page * p.page_stride);
                my_vo = pb + (OFF)off * VB;
                my_so = pb + scale_region + (OFF)off * SB;
            }
            my_out = t * p.out_stride_t + (int64_t)j * p.out_stride_j;
        }
        const int n_here = items - b0 < rpr ? (int)(items - b0) : rpr;
        for (int g = 0; g < n_here; g += GROUP) {
            uint4 raw[STEPS][CPL];     // REC 1: .x, .y = 8 value bytes; REC 2: 16 e4m3 bytes
            uint32_t scl[STEPS][CPL];  // REC 1: scale byte; REC 2: binary32 scale bits
            bool has[STEPS];
#pragma unroll
            for (int st = 0; st < STEPS; ++st) {
                const int src = g + st * GPW + grp;
                const OFF vo = shfl_off(my_vo, src);
                const OFF so = shfl_off(my_so, src);
                has[st] = vo != kZeroRow;
                if (has[st]) {
                    const uint8_t* vals = p.cache + vo;
                    const uint8_t* sc = p.cache + so;
#pragma unroll
                    for (int i = 0; i < CPL; ++i) {
                        const int c = gl + i * LANES;
                        if constexpr (REC == 1) {
                            const uint2 v = ld_nc_v2(vals + 8 * c);
                            raw[st][i].x = v.x;
                            raw[st][i].y = v.y;
                            scl[st][i] = ld_nc_u8(sc + c / 2);
                        } else {
                            raw[st][i] = ld_nc_v4(vals + 16 * c);
                            scl[st][i] = ld_nc_u32(sc);
                        }
                    }
                }
            }
#pragma unroll
            for (int st = 0; st < STEPS; ++st) {
                const int64_t off = __shfl_sync(0xFFFFFFFFu, my_out, g + st * GPW + grp);
                if (off < 0) continue;
                uint16_t* orow = p.out + off;
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    const int c = gl + i * LANES;  // values [16c, 16c + 16)
                    uint4 lo, hi;
                    if (!has[st]) {
                        lo = hi = make_uint4(0u, 0u, 0u, 0u);
                    } else if constexpr (REC == 1) {
                        const uint64_t s2 = splat_f32x2(ue8m0_scale(scl[st][i]));
                        const uint32_t a = raw[st][i].x, b = raw[st][i].y;
                        lo.x = scale_f16x2_to_bf16x2(cvt_e2m1x2_to_f16x2(a & 0xFFu), s2);
                        lo.y = scale_f16x2_to_bf16x2(cvt_e2m1x2_to_f16x2((a >> 8) & 0xFFu), s2);
                        lo.z = scale_f16x2_to_bf16x2(cvt_e2m1x2_to_f16x2((a >> 16) & 0xFFu), s2);
                        lo.w = scale_f16x2_to_bf16x2(cvt_e2m1x2_to_f16x2(a >> 24), s2);
                        hi.x = scale_f16x2_to_bf16x2(cvt_e2m1x2_to_f16x2(b & 0xFFu), s2);
                        hi.y = scale_f16x2_to_bf16x2(cvt_e2m1x2_to_f16x2((b >> 8) & 0xFFu), s2);
                        hi.z = scale_f16x2_to_bf16x2(cvt_e2m1x2_to_f16x2((b >> 16) & 0xFFu), s2);
                        hi.w = scale_f16x2_to_bf16x2(cvt_e2m1x2_to_f16x2(b >> 24), s2);
                    } else {
                        const uint64_t s2 = splat_f32x2(__uint_as_float(scl[st][i]));
                        const uint4 w = raw[st][i];
                        lo.x = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.x & 0xFFFFu), s2);
                        lo.y = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.x >> 16), s2);
                        lo.z = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.y & 0xFFFFu), s2);
                        lo.w = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.y >> 16), s2);
                        hi.x = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.z & 0xFFFFu), s2);
                        hi.y = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.z >> 16), s2);
                        hi.z = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.w & 0xFFFFu), s2);
                        hi.w = scale_f16x2_to_bf16x2(cvt_e4m3x2_to_f16x2(w.w >> 16), s2);
                    }
                    store_out32(orow + 16 * c, lo, hi, v8);
                }
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

template <int D, bool UE8M0, int SRC>
cudaError_t gather_fp8_dispatch(const ItemSource& src, int64_t items, cudaStream_t stream) {
    const int ts = D - src.g.rope_dim + 2 * src.g.rope_dim;
    constexpr int SDIM = UE8M0 ? D / 64 : 4 * (D / 64);
    // data record + the 16-byte chunks covering the scales, rounded to 16
    const int slot_bytes = (ts + ((SDIM + 15) / 16 + 1) * 16 + 15) / 16 * 16;
    const size_t smem = (size_t)kStages * kRowsPerTile * slot_bytes +
                        2 * kStages * sizeof(uint64_t) +
                        kStages * kRowsPerTile * (sizeof(int64_t) + sizeof(int32_t));
    auto kern = gather_fp8_tma_kernel<D, UE8M0, SRC>;
    static std::atomic<uint64_t> limit_set{0};
    const cudaError_t e = set_smem_limit_per_device(kern, 200 * 1024, limit_set);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTmaThreads, smem) !=
            cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t tiles = (items + kRowsPerTile - 1) / kRowsPerTile;
#ifdef PSK_GATHER_CTAS_PER_SM
    if (per_sm > PSK_GATHER_CTAS_PER_SM) per_sm = PSK_GATHER_CTAS_PER_SM;
#endif
    int64_t blocks = (int64_t)sm_count() * per_sm;
    if (blocks > tiles) blocks = tiles;
    const bool range = SRC == kSrcRange;
    const int v8 = out32_aligned(src.g.out, range ? src.r.out_stride_r : src.g.out_stride_t,
                                 range ? src.r.out_stride_i : src.g.out_stride_j);
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(kTmaThreads), smem, stream, src,
                      slot_bytes, v8);
}

template <int SRC>
cudaError_t fp8_by_dim(const ItemSource& src, int64_t items, cudaStream_t stream) {
    const bool ue = src.g.is_ue8m0 != 0;
    if (SRC >= kSrcTopk && !ue) return cudaErrorInvalidValue;  // fused forms: UE8M0 only
    switch (src.g.head_dim) {
#define PSK_FP8_CASE(DIM)                                                                  \
        case DIM:                                                                          \
            if constexpr (SRC >= kSrcTopk) return gather_fp8_dispatch<DIM, true, SRC>(src, items, stream); \
            else return ue ? gather_fp8_dispatch<DIM, true, SRC>(src, items, stream)       \
                           : gather_fp8_dispatch<DIM, false, SRC>(src, items, stream);
        PSK_FP8_CASE(64)
        PSK_FP8_CASE(128)
        PSK_FP8_CASE(256)
        PSK_FP8_CASE(512)
        PSK_FP8_CASE(1024)
#undef PSK_FP8_CASE
        default: return cudaErrorInvalidValue;
    }
}

#ifndef PSK_SMALL_RPR
#define PSK_SMALL_RPR 0  // items a warp resolves per round; 0: chosen per launch
#endif

template <int D, int REC, int SRC, typename OFF>
cudaError_t gather_small_launch(const GatherParams& p, const TopkSource& tk,
                                cudaStream_t stream) {
    constexpr int LANES = (D / 16) < kWarp ? (D / 16) : kWarp;
    constexpr int GPW = kWarp / LANES;
    constexpr int STEPS = (kWarp / GPW) < kSmallSteps ? (kWarp / GPW) : kSmallSteps;
    constexpr int GROUP = STEPS * GPW;
    auto kern = gather_small_kernel<D, REC, SRC, OFF>;
    const int64_t items = p.rows * (int64_t)p.cols;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t resident_warps = (int64_t)sm_count() * per_sm * (kThreads / kWarp);
    // Items per warp round: 32 (one per lane, the fewest instructions per row)
    // when the batch still gives every resident warp a full round, else fewer,
    // so that small batches keep every warp's loads in flight.  Measured alone
    // (events, L2 flushed): the 8.4 M-row prefill gather 411.7 / 397.3 /
    // 387.1 us at 8 / 16 / 32 items per round, the 262,144-row MXFP4 batch
    // 20.5 / 20.5 / 18.4 us, the 32,768-row decode batch 8.2 / 10.2 / 14.3 us.
    int rpr = GROUP;
    while (rpr < kWarp && items >= (int64_t)2 * rpr * resident_warps) rpr *= 2;
    if (PSK_SMALL_RPR > 0) rpr = PSK_SMALL_RPR;
    const int64_t warps = (items + rpr - 1) / rpr;
    const int64_t need = (warps * kWarp + kThreads - 1) / kThreads;
    const int64_t full = (int64_t)sm_count() * per_sm;
    const int64_t blocks = need < full ? need : full;
    const int v8 = out32_aligned(p.out, p.out_stride_t, p.out_stride_j);
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), 0, stream, p, tk, rpr, v8);
}

template <int D, int REC, int SRC>
cudaError_t gather_small_dispatch(const GatherParams& p, const TopkSource& tk,
                                  cudaStream_t stream) {
    // 32-bit record offsets while every byte of the cache is below 4 GiB
    if (p.num_pages * p.page_stride < (int64_t(1) << 32) - 1)
        return gather_small_launch<D, REC, SRC, uint32_t>(p, tk, stream);
    return gather_small_launch<D, REC, SRC, uint64_t>(p, tk, stream);
}

template <int REC, int SRC>
cudaError_t gather_small_by_dim(const GatherParams& p, const TopkSource& tk, cudaStream_t stream) {
    switch (p.head_dim) {
        case 32: return gather_small_dispatch<32, REC, SRC>(p, tk, stream);
        case 64: return gather_small_dispatch<64, REC, SRC>(p, tk, stream);
        case 128: return gather_small_dispatch<128, REC, SRC>(p, tk, stream);
        case 256: return gather_small_dispatch<256, REC, SRC>(p, tk, stream);
        case 512: return gather_small_dispatch<512, REC, SRC>(p, tk, stream);
        case 1024: return gather_small_dispatch<1024, REC, SRC>(p, tk, stream);
        default: return cudaErrorInvalidValue;
    }
}

// Failure-path check of the bounded wait: one thread waits on a barrier that
// nothing completes, gives up after limit_ns and counts the expiry exactly as
// the pipelined kernels do; the kernel then returns normally.
__global__ void wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    mbar_fence_init();
    if (!mbar_wait_bounded(&bar, 0, limit_ns)) atomicAdd(&g_wait_timeouts, 1u);
}

}  // namespace

cudaError_t read_wait_timeouts(uint32_t* count) {
    return cudaMemcpyFromSymbol(count, g_wait_timeouts, sizeof(uint32_t));
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, kWarp, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_gather(const GatherParams& params, cudaStream_t stream) {
    GatherParams p = params;
    p.block_shift = log2_if_pow2(p.block_size);
    if (p.record == 0) {
        ItemSource src{};
        src.g = p;
        return fp8_by_dim<kSrcIndex>(src, p.rows * (int64_t)p.cols, stream);
    }
    const TopkSource none{};
    return p.record == 1 ? gather_small_by_dim<1, kSrcIndex>(p, none, stream)
                         : gather_small_by_dim<2, kSrcIndex>(p, none, stream);
}

cudaError_t launch_gather_topk(const GatherParams& params, const TopkSource& tk,
                               cudaStream_t stream) {
    GatherParams p = params;
    p.block_shift = log2_if_pow2(p.block_size);
    if (p.record == 0) {
        ItemSource src{};
        src.g = p;
        src.tk = tk;
        return fp8_by_dim<kSrcTopk>(src, p.rows * (int64_t)p.cols, stream);
    }
    return p.record == 1 ? gather_small_by_dim<1, kSrcTopk>(p, tk, stream)
                         : gather_small_by_dim<2, kSrcTopk>(p, tk, stream);
}

cudaError_t launch_gather_window(const GatherParams& params, const WindowSource& wn,
                                 cudaStream_t stream) {
    GatherParams p = params;
    p.block_shift = log2_if_pow2(p.block_size);
    if (p.record != 0) return cudaErrorInvalidValue;
    ItemSource src{};
    src.g = p;
    src.wn = wn;
    return fp8_by_dim<kSrcWindow>(src, p.rows * (int64_t)p.cols, stream);
}

cudaError_t launch_gather_pair(const GatherParams& params, const PairSource& pr,
                               cudaStream_t stream) {
    GatherParams p = params;
    p.block_shift = log2_if_pow2(p.block_size);
    if (p.record != 0) return cudaErrorInvalidValue;
    ItemSource src{};
    src.g = p;
    src.pr = pr;
    src.pr.block_shift = log2_if_pow2(pr.block_size);
    return fp8_by_dim<kSrcPair>(src, p.rows * (int64_t)p.cols, stream);
}

cudaError_t launch_gather_dense(const GatherParams& params, const DenseSource& ds,
                                cudaStream_t stream) {
    GatherParams p = params;
    p.block_shift = log2_if_pow2(p.block_size);
    if (p.record != 0) return cudaErrorInvalidValue;
    ItemSource src{};
    src.g = p;
    src.ds = ds;
    return fp8_by_dim<kSrcDense>(src, p.rows * (int64_t)p.cols, stream);
}

cudaError_t launch_gather_ranges(const RangeParams& r, cudaStream_t stream) {
    ItemSource src{};
    src.r = r;
    src.g.out = r.out;
    src.g.cache = r.cache;
    src.g.num_pages = r.num_pages;
    src.g.page_stride = r.page_stride;
    src.g.block_size = r.block_size;
    src.g.block_shift = log2_if_pow2(r.block_size);
    src.g.record = 0;
    src.g.head_dim = r.head_dim;
    src.g.rope_dim = r.rope_dim;
    src.g.is_ue8m0 = r.is_ue8m0;
    return fp8_by_dim<kSrcRange>(src, (int64_t)r.num_reqs * (r.out_rows - r.offset), stream);
}

// ---- raw MXFP4 paged gather ----------------------------------------------------------
//
// TokenSpeed models/deepseek_v4.py, _deepseek_v4_gather_paged_indexer_mxfp4_cache
// (indexer_mxfp4_paged_gather): packed records copied unchanged, request r's
// local positions 0.. to output rows cu_seq_lens[r]..  A group of D/8 lanes
// (at most 32) owns one row: each lane copies 4 value bytes, lane 0 the scale
// bytes.  A row finds its request by binary search over cu_seq_lens.
template <int D>
__global__ void __launch_bounds__(kThreads) mxfp4_raw_gather_kernel(RawGatherParams p) {
    constexpr int CHUNKS = D / 8;  // 4 value bytes per chunk
    constexpr int LANES = CHUNKS < kWarp ? CHUNKS : kWarp;
    constexpr int CPL = CHUNKS / LANES;
    constexpr int VB = D / 2, SB = D / 32;
    const int lane = threadIdx.x & 31;
    const int gl = lane % LANES;
    const int64_t gid = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / LANES;
    const int64_t ngroups = (int64_t)gridDim.x * kThreads / LANES;
    const int64_t capacity = p.num_pages * (int64_t)p.block_size;
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t row = gid; row < p.total_rows; row += ngroups) {
        // last request r with cu_seq_lens[r] <= row
        int lo = 0, hi = p.num_reqs;  // invariant: cu[lo] <= row (when valid)
        while (hi - lo > 1) {
            const int mid = (lo + hi) / 2;
            if ((int64_t)__ldg(p.cu_seq_lens + mid) <= row) lo = mid; else hi = mid;
        }
        const int64_t start = __ldg(p.cu_seq_lens + lo), end = __ldg(p.cu_seq_lens + lo + 1);
        int32_t s = -1;
        if (row >= start && row < end) {
            const int64_t i = row - start;
            int64_t rem;
            const int64_t lp = div_block(i, p.block_size, p.block_shift, rem);
            if (lp < p.bt_width) {
                const int32_t page = __ldg(p.block_table + (int64_t)lo * p.bt_stride + lp);
                if (page >= 0) {
                    const int64_t sl = (int64_t)page * p.block_size + rem;
                    if (sl < capacity) s = (int32_t)sl;
                }
            }
        }
        uint8_t* vo = p.values_out + row * VB;
        uint8_t* so = p.scales_out + row * SB;
        if (s < 0) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) *reinterpret_cast<uint32_t*>(vo + 4 * (gl + c * LANES)) = 0u;
            if (gl == 0) for (int b = 0; b < SB; ++b) so[b] = 0;
            continue;
        }
        int32_t off;
        const int32_t page = div_block32(s, p.block_size, p.block_shift, off);
        const uint8_t* base = p.cache + (int64_t)page * p.page_stride;
        const uint8_t* vals = base + (int64_t)off * VB;
        const uint8_t* scl = base + (int64_t)p.block_size * VB + (int64_t)off * SB;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int k = gl + c * LANES;
            *reinterpret_cast<uint32_t*>(vo + 4 * k) = ld_nc_u32(vals + 4 * k);
        }
        if (gl == 0) {
            if (SB % 4 == 0) {
                for (int b = 0; b < SB; b += 4)
                    *reinterpret_cast<uint32_t*>(so + b) = ld_nc_u32(scl + b);
            } else {
                for (int b = 0; b < SB; ++b) so[b] = (uint8_t)ld_nc_u8(scl + b);
            }
        }
    }
}

template <int D>
cudaError_t raw_dispatch(const RawGatherParams& p, cudaStream_t stream) {
    constexpr int LANES = (D / 8) < kWarp ? (D / 8) : kWarp;
    auto kern = mxfp4_raw_gather_kernel<D>;
    const int64_t blocks = persistent_blocks(kern, p.total_rows, LANES);
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), 0, stream, p);
}

cudaError_t launch_mxfp4_raw_gather(const RawGatherParams& params, cudaStream_t stream) {
    RawGatherParams p = params;
    p.block_shift = log2_if_pow2(p.block_size);
    switch (p.head_dim) {
        case 32: return raw_dispatch<32>(p, stream);
        case 64: return raw_dispatch<64>(p, stream);
        case 128: return raw_dispatch<128>(p, stream);
        case 256: return raw_dispatch<256>(p, stream);
        case 512: return raw_dispatch<512>(p, stream);
        case 1024: return raw_dispatch<1024>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace psk
