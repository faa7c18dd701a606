// gather.h -- parameters and launchers of the dequantize-and-gather kernels (internal).
#pragma once

#include "launch.h"

namespace psk {

struct GatherParams {
    uint16_t* out;
    int64_t out_stride_t;
    int64_t out_stride_j;
    const uint8_t* cache;
    int64_t num_pages;
    int64_t page_stride;
    int32_t block_size;
    int32_t record;
    int32_t head_dim;
    int32_t rope_dim;
    int32_t is_ue8m0;
    const int32_t* idx;
    int64_t idx_stride;
    int64_t rows;
    int32_t cols;
    int32_t block_shift;  // log2(block_size) or -1; set by the launcher
};

cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream);

// Range form: per request r, rows i < out_rows - offset; g = gather_lens[r]
// (or seq_lens[r]); row i < g is position seq_lens[r] - g + i -> out row
// offset + i; rows i >= g are not written.
struct RangeParams {
    uint16_t* out;
    int64_t out_stride_r;
    int64_t out_stride_i;
    int64_t out_rows;
    int64_t offset;
    const uint8_t* cache;
    int64_t num_pages;
    int64_t page_stride;
    int32_t block_size;
    int32_t head_dim;
    int32_t rope_dim;
    int32_t is_ue8m0;
    const int32_t* seq_lens;
    const int32_t* gather_lens;
    const int32_t* block_table;
    int64_t bt_stride;
    int32_t bt_width;
    const int32_t* base_offsets;
    int32_t num_reqs;
};

cudaError_t launch_gather_ranges(const RangeParams& p, cudaStream_t stream);

struct RawGatherParams {
    uint8_t* values_out;
    uint8_t* scales_out;
    const uint8_t* cache;
    int64_t num_pages;
    int64_t page_stride;
    int32_t block_size;
    int32_t head_dim;
    const int32_t* block_table;
    int64_t bt_stride;
    int32_t bt_width;
    const int32_t* cu_seq_lens;
    int32_t num_reqs;
    int64_t total_rows;
    int32_t block_shift;  // log2(block_size) or -1; set by the launcher
};

cudaError_t launch_mxfp4_raw_gather(const RawGatherParams& p, cudaStream_t stream);

// Number of bounded in-kernel waits that expired on the current device.

// Slots computed in the gather itself (no index matrix): the top-k columns of
// a token (a local top-k index through the request's table, the
// compute_global_topk_indices_and_lens rule) or its window columns (the
// window rule of combine_topk_swa_indices through the SWA table).
struct TopkSource {
    const int32_t* topk_local;  // [rows, topk_stride]
    int64_t topk_stride;
    const int32_t* t2r;
    const uint8_t* valid;       // nullable
    int32_t num_reqs;
    const int32_t* bt;
    int64_t bt_stride;
    int32_t bt_width;
    const int32_t* base;        // nullable
};

struct WindowSource {
    const int32_t* qsl;
    const int32_t* seq_lens;
    const int32_t* t2r;
    const int32_t* replay;      // nullable
    const uint8_t* valid;       // nullable
    int32_t num_reqs;
    const int32_t* bt;
    int64_t bt_stride;
    int32_t bt_width;
    const int32_t* base;        // nullable
};

// p.idx is unused: rows = tokens, cols = topk (or window); out as in p.
// Two caches of one record format read through one index matrix: columns
// j >= split take their slots in this cache, columns j < split in GatherParams'.
struct PairSource {
    const uint8_t* cache;
    int64_t num_pages;
    int64_t page_stride;
    int32_t block_size;
    int32_t block_shift;  // set by the launcher
    int32_t split;
};

cudaError_t launch_gather_pair(const GatherParams& p, const PairSource& s, cudaStream_t stream);

// Every visible compressed entry of a token (the HCA decode rule): entry c of
// token t is compressed position c when c < clamp(floor((positions[t] + 1) /
// ratio), 0, cols), mapped through its request's table.
struct DenseSource {
    const int64_t* positions;
    const int32_t* t2r;
    const uint8_t* valid;   // may be null
    int32_t num_reqs;
    const int32_t* bt;
    int64_t bt_stride;
    int32_t bt_width;
    const int32_t* base;    // may be null
    int32_t ratio;
};

cudaError_t launch_gather_dense(const GatherParams& p, const DenseSource& s, cudaStream_t stream);
cudaError_t launch_gather_topk(const GatherParams& p, const TopkSource& s, cudaStream_t stream);
cudaError_t launch_gather_window(const GatherParams& p, const WindowSource& s,
                                 cudaStream_t stream);

// Count of expired bounded waits in the gather kernels.
cudaError_t read_wait_timeouts(uint32_t* count);

// One bounded wait on a barrier nothing completes (counted when it expires).
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream);

}  // namespace psk
