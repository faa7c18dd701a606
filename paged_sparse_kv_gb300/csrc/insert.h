// insert.h -- parameters and launchers of the quantize-and-insert kernels (internal).
#pragma once

#include "launch.h"

namespace psk {

struct InsertParams {
    const void* k;
    int64_t k_row_stride;
    const int64_t* slots;
    int64_t num_tokens;
    uint8_t* cache;
    int64_t num_pages;
    int64_t page_stride;
    int32_t block_size;
    int32_t head_dim;
    int32_t rope_dim;   // fp8 record only
    int32_t is_ue8m0;   // fp8 record only
    int32_t* err_count;
};

cudaError_t launch_fp8_insert(const InsertParams& p, cudaStream_t stream);
cudaError_t launch_mxfp4_insert(const InsertParams& p, cudaStream_t stream);
// The FP8 indexer record (per-token power-of-two binary32 scale).
cudaError_t launch_fp8_indexer_insert(const InsertParams& p, cudaStream_t stream);

// indexer_k_norm_rope_store: 128-dim keys, RMSNorm -> GPT-J RoPE on the last
// 64 dims -> MXFP4 or FP8 indexer record -> paged store.
struct NormRopeParams {
    const uint16_t* k;        // bf16 [num_tokens, k_row_stride]
    int64_t k_row_stride;
    const int64_t* positions;
    const float* cos_sin;     // [max_pos, cs_stride]: 32 cos then 32 sin
    int64_t cs_stride;
    int64_t max_pos;
    const float* weight;      // [128]
    float eps;
    const int64_t* slots;
    int64_t num_tokens;
    int32_t ratio;
    int32_t record;           // 1 = MXFP4, 2 = FP8 indexer
    uint8_t* cache;
    int64_t num_pages;
    int64_t page_stride;
    int32_t block_size;
    int32_t* err_count;
    int32_t ratio_shift;      // log2(ratio) for a power-of-two ratio, else -1 (launcher)
};

cudaError_t launch_norm_rope_store(const NormRopeParams& p, cudaStream_t stream);

}  // namespace psk
