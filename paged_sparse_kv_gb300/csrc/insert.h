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

}  // namespace psk
