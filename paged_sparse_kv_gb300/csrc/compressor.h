// compressor.h -- parameters and launchers of the compressed-KV producer (internal).
#pragma once

#include "launch.h"

namespace psk {

struct SaveStateParams {
    const float* kv;          // [num_tokens, in_stride]
    const float* score;       // [num_tokens, in_stride]
    int64_t in_stride;
    const float* ape;         // [ratio, state_width]
    int32_t state_width;
    const int64_t* slots;
    const int64_t* positions;
    int64_t num_tokens;
    int32_t ratio;
    float* state;             // [num_pages, block_size, 2 * state_width]
    int64_t num_pages;
    int32_t block_size;
    int32_t* err_count;
};

cudaError_t launch_save_compressor_state(const SaveStateParams& p, cudaStream_t stream);

struct CompressParams {
    const float* state;       // [state_pages, state_bs, 2 * state_width]
    int64_t state_pages;
    int32_t state_bs;
    int32_t state_width;
    const int32_t* t2r;
    const int64_t* positions;
    const int64_t* state_slots;
    const int32_t* bt;
    int64_t bt_stride;
    int32_t bt_width;
    const int32_t* base;
    int32_t num_reqs;
    int64_t num_tokens;
    int32_t ratio;
    int32_t overlap;
    const float* weight;      // [512]
    float eps;
    const float* cos_sin;     // [max_pos, cs_stride]
    int64_t cs_stride;
    int64_t max_pos;
    uint8_t* kv_cache;
    int64_t kv_pages;
    int64_t kv_page_stride;
    int32_t kv_bs;
    const int64_t* kv_slots;
    int32_t* err_count;
};

cudaError_t launch_compress_kv_insert(const CompressParams& p, cudaStream_t stream);

// Copies of the long-window kernel whose bounded wait gave up.
cudaError_t read_compress_wait_timeouts(uint32_t* count);

}  // namespace psk
