// index_build.h -- parameters and launchers of the index builders (internal).
#pragma once

#include "launch.h"

namespace psk {

struct IndexParams {
    const int32_t* qsl;
    const int32_t* seq_lens;
    const int32_t* t2r;
    const int32_t* replay;
    int32_t num_reqs;
    int64_t num_tokens;
    const int32_t* swa_bt;
    int64_t swa_stride;
    int32_t swa_width;
    const int32_t* swa_base;
    int32_t swa_bs;
    int32_t swa_shift;   // log2(swa_bs) or -1
    const int32_t* comp_bt;
    int64_t comp_stride;
    int32_t comp_width;
    const int32_t* comp_base;
    int32_t comp_bs;
    int32_t comp_shift;
    int32_t window;
    int32_t topk;
    int32_t out_cols;
    const int32_t* topk_local;
    int64_t topk_stride;
    const uint8_t* valid;
    int32_t* out;
    int64_t out_stride;
    int32_t* lens;
    // launch shape, filled by the launcher
    int32_t tokens_per_cta;
    int32_t warps_per_token;
    int32_t stage_comp;  // entries of the compressed row staged in shared memory
    int32_t stage_swa;   // entries of the SWA row staged in shared memory
    int32_t swa_maxp, swa_maxrem;    // INT32_MAX / swa_bs, INT32_MAX % swa_bs
    int32_t comp_maxp, comp_maxrem;  // the same for comp_bs
};

// has_swa = true: the fused window + top-k build; false: top-k mapping only.
cudaError_t launch_index_build(IndexParams p, bool has_swa, cudaStream_t stream);

struct WorkspaceIndexParams {
    const int32_t* qsl;
    const int32_t* seq_lens;
    const int32_t* gather_lens;
    const int32_t* t2r;
    int32_t num_reqs;
    int64_t num_tokens;
    int32_t window;
    int32_t compress_ratio;
    const int32_t* topk_local;
    int64_t topk_stride;
    int32_t topk;
    int64_t workspace_width;
    int64_t compressed_base;
    const uint8_t* valid;
    int32_t* out;
    int64_t out_stride;
    int32_t* lens;
    const int64_t* positions;  // non-null: token positions given (qsl unused)
};

cudaError_t launch_workspace_indices(const WorkspaceIndexParams& p, cudaStream_t stream);

// Dense builders: every visible compressed entry of a token (HCA decode:
// slots through the table + lens; prefill: request-local entry numbers).
struct DenseParams {
    const int64_t* positions;
    int64_t num_tokens;
    const int32_t* t2r;      // global form only
    int32_t num_reqs;
    const int32_t* bt;       // global form only
    int64_t bt_stride;
    int32_t bt_width;
    const int32_t* base;
    int32_t bs;
    int32_t ratio;
    int32_t width;
    const uint8_t* valid;
    int32_t* out;
    int64_t out_stride;
    int32_t* lens;           // global form only
};

// global = true: compute_dense_compressed_indices_and_lens; false:
// build_dense_prefill_local_compressed_indices.
cudaError_t launch_dense_indices(const DenseParams& p, bool global, cudaStream_t stream);

// Count of expired bounded waits in the index builders.
cudaError_t read_index_wait_timeouts(uint32_t* count);

}  // namespace psk
