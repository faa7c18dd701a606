// launch.h -- host-side launchers behind the libpsk C ABI (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace psk {

// Launch with programmatic stream serialisation (PDL): the kernel may begin
// while its predecessor on the stream finishes; it calls pdl_wait() before
// touching global memory.  Inside a CUDA graph this becomes a programmatic
// edge.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Number of SMs on the current device (queried once per device).
int sm_count();

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
cudaError_t read_wait_timeouts(uint32_t* count);        // gather kernels
cudaError_t read_index_wait_timeouts(uint32_t* count);  // index builders

}  // namespace psk
