// abi.cu -- the extern "C" entry points of libpsk (declared in include/psk.h).
//
// Each entry point validates its arguments on the host, returns
// PSK_ERR_INVALID_ARGUMENT before touching the GPU when they are wrong,
// returns PSK_OK without a launch when there is no work, and otherwise
// launches exactly one kernel on the caller's stream.  Nothing here
// allocates, synchronises or keeps state beyond the per-thread error text.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "compressor.h"
#include "gather.h"
#include "index_build.h"
#include "insert.h"
#include "launch.h"
#include "psk.h"
#include "psk_common.cuh"

namespace {

thread_local std::string g_last_error;

psk_status fail(psk_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

psk_status ok() {
    g_last_error.clear();
    return PSK_OK;
}

psk_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return ok();
    return fail(PSK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

#define CHECK(cond, ...)                                                \
    do {                                                                \
        if (!(cond)) return fail(PSK_ERR_INVALID_ARGUMENT, __VA_ARGS__); \
    } while (0)

bool fp8_head_dim_ok(int32_t d) { return d == 64 || d == 128 || d == 256 || d == 512 || d == 1024; }
bool mxfp4_head_dim_ok(int32_t d) {
    return d == 32 || d == 64 || d == 128 || d == 256 || d == 512 || d == 1024;
}

int64_t fp8_record_bytes(int32_t head_dim, int32_t rope_dim, int32_t ue8m0) {
    return (int64_t)(head_dim - rope_dim) + 2 * (int64_t)rope_dim +
           (int64_t)(head_dim / 64) * (ue8m0 ? 1 : 4);
}

psk_status check_cache(const uint8_t* cache, int64_t num_pages, int64_t page_stride,
                       int32_t block_size, int64_t record_bytes) {
    CHECK(cache != nullptr, "cache is null");
    CHECK(num_pages >= 1, "num_pages must be >= 1 (got %lld)", (long long)num_pages);
    CHECK(block_size >= 1, "block_size must be >= 1 (got %d)", block_size);
    CHECK(page_stride >= (int64_t)block_size * record_bytes,
          "page_stride %lld is smaller than block_size * record bytes = %lld",
          (long long)page_stride, (long long)block_size * record_bytes);
    CHECK(page_stride % 16 == 0, "page_stride must be a multiple of 16 bytes");
    CHECK(aligned(cache, 16), "cache must be 16-byte aligned");
    CHECK(num_pages <= INT64_MAX / page_stride, "cache size overflows int64");
    return PSK_OK;
}

}  // namespace

extern "C" {

const char* psk_last_error(void) { return g_last_error.c_str(); }

int32_t psk_abi_version(void) { return 5; }

psk_status psk_device_wait_timeouts(uint32_t* count) {
    CHECK(count != nullptr, "count must be non-null");
    uint32_t gather = 0, index = 0, compress = 0;
    psk_status st = cuda_status(psk::read_wait_timeouts(&gather), "reading the wait-timeout counter");
    if (st != PSK_OK) return st;
    st = cuda_status(psk::read_index_wait_timeouts(&index), "reading the wait-timeout counter");
    if (st != PSK_OK) return st;
    st = cuda_status(psk::read_compress_wait_timeouts(&compress), "reading the wait-timeout counter");
    if (st != PSK_OK) return st;
    *count = gather + index + compress;
    return PSK_OK;
}

psk_status psk_device_wait_selftest(uint64_t limit_ns, psk_stream_t stream) {
    CHECK(limit_ns >= 1000 && limit_ns <= 1000000000ull, "limit_ns must be in [1e3, 1e9]");
    return cuda_status(psk::launch_wait_selftest(limit_ns, reinterpret_cast<cudaStream_t>(stream)),
                       "psk_device_wait_selftest launch");
}

psk_status quantize_and_insert_k_cache(const void* k, int64_t k_row_stride,
                                       const int64_t* slot_mapping, int64_t num_tokens,
                                       uint8_t* k_cache, int64_t num_pages, int64_t page_stride,
                                       int32_t block_size, int32_t head_dim, int32_t rope_dim,
                                       int32_t is_ue8m0, int32_t* err_count,
                                       psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(is_ue8m0 == 0 || is_ue8m0 == 1, "is_ue8m0 must be 0 or 1");
    CHECK(fp8_head_dim_ok(head_dim), "head_dim must be one of 64, 128, 256, 512, 1024 (got %d)",
          head_dim);
    CHECK(rope_dim >= 0 && rope_dim < head_dim && rope_dim % 64 == 0,
          "rope_dim must be a multiple of 64 in [0, head_dim) (got %d)", rope_dim);
    psk_status st = check_cache(k_cache, num_pages, page_stride, block_size,
                                fp8_record_bytes(head_dim, rope_dim, is_ue8m0));
    if (st != PSK_OK) return st;
    if (num_tokens == 0) return ok();
    CHECK(k != nullptr && slot_mapping != nullptr, "k and slot_mapping must be non-null");
    CHECK(aligned(k, 16), "k must be 16-byte aligned");
    CHECK(k_row_stride >= head_dim && k_row_stride % 8 == 0,
          "k_row_stride must be >= head_dim and a multiple of 8 elements");
    CHECK(aligned(slot_mapping, 8), "slot_mapping must be 8-byte aligned");
    CHECK(err_count == nullptr || aligned(err_count, 4), "err_count must be 4-byte aligned");
    psk::InsertParams p{k, k_row_stride, slot_mapping, num_tokens, k_cache, num_pages,
                        page_stride, block_size, head_dim, rope_dim, is_ue8m0, err_count};
    return cuda_status(psk::launch_fp8_insert(p, reinterpret_cast<cudaStream_t>(stream)),
                       "quantize_and_insert_k_cache launch");
}

psk_status write_indexer_mxfp4_cache(const void* index_k, int64_t k_row_stride,
                                     const int64_t* slot_mapping, int64_t num_tokens,
                                     uint8_t* cache, int64_t num_pages, int64_t page_stride,
                                     int32_t block_size, int32_t head_dim, int32_t* err_count,
                                     psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(mxfp4_head_dim_ok(head_dim),
          "head_dim must be one of 32, 64, 128, 256, 512, 1024 (got %d)", head_dim);
    psk_status st = check_cache(cache, num_pages, page_stride, block_size,
                                head_dim / 2 + head_dim / 32);
    if (st != PSK_OK) return st;
    if (num_tokens == 0) return ok();
    CHECK(index_k != nullptr && slot_mapping != nullptr,
          "index_k and slot_mapping must be non-null");
    CHECK(aligned(index_k, 16), "index_k must be 16-byte aligned");
    CHECK(k_row_stride >= head_dim && k_row_stride % 8 == 0,
          "k_row_stride must be >= head_dim and a multiple of 8 elements");
    CHECK(aligned(slot_mapping, 8), "slot_mapping must be 8-byte aligned");
    CHECK(err_count == nullptr || aligned(err_count, 4), "err_count must be 4-byte aligned");
    psk::InsertParams p{index_k, k_row_stride, slot_mapping, num_tokens, cache, num_pages,
                        page_stride, block_size, head_dim, 0, 1, err_count};
    return cuda_status(psk::launch_mxfp4_insert(p, reinterpret_cast<cudaStream_t>(stream)),
                       "write_indexer_mxfp4_cache launch");
}

psk_status compute_global_topk_indices_and_lens(
    const int32_t* topk_local, int64_t topk_stride, int64_t num_tokens, int32_t topk,
    const int32_t* token_to_req, const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    int32_t num_reqs, int32_t block_size, const int32_t* base_offsets,
    const uint8_t* is_valid_token, int32_t* out_indices, int64_t out_stride, int32_t* out_lens,
    psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(topk >= 0, "topk must be >= 0");
    CHECK(block_size >= 1, "block_size must be >= 1");
    CHECK(bt_width >= 0 && bt_stride >= bt_width, "need 0 <= bt_width <= bt_stride");
    CHECK(topk_stride >= topk && out_stride >= topk, "row strides must be >= topk");
    if (num_tokens == 0) return ok();
    CHECK(num_reqs >= 1, "num_reqs must be >= 1");
    CHECK(token_to_req && out_lens, "token_to_req and out_lens must be non-null");
    CHECK(topk == 0 || (topk_local && out_indices), "topk_local and out_indices must be non-null");
    CHECK(bt_width == 0 || block_table, "block_table must be non-null");
    CHECK(aligned(topk_local, 4) && aligned(out_indices, 4) && aligned(token_to_req, 4) &&
              aligned(block_table, 4) && aligned(base_offsets, 4) && aligned(out_lens, 4),
          "int32 arrays must be 4-byte aligned");
    psk::IndexParams p{};
    p.t2r = token_to_req;
    p.num_reqs = num_reqs;
    p.num_tokens = num_tokens;
    p.comp_bt = block_table;
    p.comp_stride = bt_stride;
    p.comp_width = bt_width;
    p.comp_base = base_offsets;
    p.comp_bs = block_size;
    p.comp_shift = psk::log2_if_pow2(block_size);
    p.window = 0;
    p.topk = topk;
    p.out_cols = topk;
    p.topk_local = topk_local;
    p.topk_stride = topk_stride;
    p.valid = is_valid_token;
    p.out = out_indices;
    p.out_stride = out_stride;
    p.lens = out_lens;
    return cuda_status(psk::launch_index_build(p, false, reinterpret_cast<cudaStream_t>(stream)),
                       "compute_global_topk_indices_and_lens launch");
}

psk_status combine_topk_swa_indices(
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* token_to_req,
    const int32_t* replay_start, int32_t num_reqs, int64_t num_tokens,
    const int32_t* swa_block_table, int64_t swa_bt_stride, int32_t swa_bt_width,
    const int32_t* swa_base_offsets, int32_t swa_block_size, const int32_t* comp_block_table,
    int64_t comp_bt_stride, int32_t comp_bt_width, const int32_t* comp_base_offsets,
    int32_t comp_block_size, int32_t window, int32_t compress_ratio, const int32_t* topk_local,
    int64_t topk_stride, int32_t topk, const uint8_t* is_valid_token, int32_t* sparse_indices,
    int64_t out_stride, int32_t* lens, psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(window >= 0 && topk >= 0, "window and topk must be >= 0");
    CHECK(compress_ratio >= 1, "compress_ratio must be >= 1");
    CHECK(swa_block_size >= 1 && comp_block_size >= 1, "block sizes must be >= 1");
    CHECK(swa_bt_width >= 0 && swa_bt_stride >= swa_bt_width,
          "need 0 <= swa_bt_width <= swa_bt_stride");
    if (comp_block_table != nullptr) {
        CHECK(comp_bt_width >= 0 && comp_bt_stride >= comp_bt_width,
              "need 0 <= comp_bt_width <= comp_bt_stride");
    }
    const int64_t padded = ((int64_t)topk + 3) / 4 * 4;
    const int64_t cols = (int64_t)window + padded;
    CHECK(cols <= INT32_MAX, "window + padded topk overflows int32");
    CHECK(topk_stride >= topk, "topk_stride must be >= topk");
    CHECK(out_stride >= cols, "out_stride must be >= window + roundup(topk, 4)");
    if (num_tokens == 0) return ok();
    CHECK(num_reqs >= 1, "num_reqs must be >= 1");
    CHECK(query_start_loc && seq_lens && token_to_req && sparse_indices && lens,
          "query_start_loc, seq_lens, token_to_req, sparse_indices and lens must be non-null");
    CHECK(topk == 0 || topk_local, "topk_local must be non-null");
    CHECK(swa_bt_width == 0 || swa_block_table, "swa_block_table must be non-null");
    CHECK(aligned(query_start_loc, 4) && aligned(seq_lens, 4) && aligned(token_to_req, 4) &&
              aligned(replay_start, 4) && aligned(swa_block_table, 4) &&
              aligned(swa_base_offsets, 4) && aligned(comp_block_table, 4) &&
              aligned(comp_base_offsets, 4) && aligned(topk_local, 4) &&
              aligned(sparse_indices, 4) && aligned(lens, 4),
          "int32 arrays must be 4-byte aligned");
    psk::IndexParams p{};
    p.qsl = query_start_loc;
    p.seq_lens = seq_lens;
    p.t2r = token_to_req;
    p.replay = replay_start;
    p.num_reqs = num_reqs;
    p.num_tokens = num_tokens;
    p.swa_bt = swa_block_table;
    p.swa_stride = swa_bt_stride;
    p.swa_width = swa_bt_width;
    p.swa_base = swa_base_offsets;
    p.swa_bs = swa_block_size;
    p.swa_shift = psk::log2_if_pow2(swa_block_size);
    if (comp_block_table == nullptr) {
        p.comp_bt = swa_block_table;
        p.comp_stride = swa_bt_stride;
        p.comp_width = swa_bt_width;
    } else {
        p.comp_bt = comp_block_table;
        p.comp_stride = comp_bt_stride;
        p.comp_width = comp_bt_width;
    }
    p.comp_base = comp_base_offsets;
    p.comp_bs = comp_block_size;
    p.comp_shift = psk::log2_if_pow2(comp_block_size);
    p.window = window;
    p.topk = topk;
    p.out_cols = (int32_t)cols;
    p.topk_local = topk_local;
    p.topk_stride = topk_stride;
    p.valid = is_valid_token;
    p.out = sparse_indices;
    p.out_stride = out_stride;
    p.lens = lens;
    return cuda_status(psk::launch_index_build(p, true, reinterpret_cast<cudaStream_t>(stream)),
                       "combine_topk_swa_indices launch");
}

psk_status dequantize_and_gather_k_cache(void* out, int64_t out_stride_t, int64_t out_stride_j,
                                         const uint8_t* cache, int64_t num_pages,
                                         int64_t page_stride, int32_t block_size,
                                         psk_record record, int32_t head_dim, int32_t rope_dim,
                                         int32_t is_ue8m0, const int32_t* indices,
                                         int64_t idx_stride, int64_t rows, int32_t cols,
                                         psk_stream_t stream) {
    CHECK(rows >= 0 && cols >= 0, "rows and cols must be >= 0");
    CHECK(record == PSK_REC_FP8_DS_MLA || record == PSK_REC_MXFP4 ||
              record == PSK_REC_FP8_INDEXER,
          "unknown record %d", (int)record);
    int64_t rec_bytes;
    if (record == PSK_REC_FP8_INDEXER) {
        CHECK(mxfp4_head_dim_ok(head_dim),
              "head_dim must be one of 32, 64, 128, 256, 512, 1024 (got %d)", head_dim);
        CHECK(rope_dim == 0, "rope_dim must be 0 for the FP8 indexer record");
        rec_bytes = head_dim + 4;
    } else if (record == PSK_REC_FP8_DS_MLA) {
        CHECK(is_ue8m0 == 0 || is_ue8m0 == 1, "is_ue8m0 must be 0 or 1");
        CHECK(fp8_head_dim_ok(head_dim),
              "head_dim must be one of 64, 128, 256, 512, 1024 (got %d)", head_dim);
        CHECK(rope_dim >= 0 && rope_dim < head_dim && rope_dim % 64 == 0,
              "rope_dim must be a multiple of 64 in [0, head_dim) (got %d)", rope_dim);
        rec_bytes = fp8_record_bytes(head_dim, rope_dim, is_ue8m0);
    } else {
        CHECK(mxfp4_head_dim_ok(head_dim),
              "head_dim must be one of 32, 64, 128, 256, 512, 1024 (got %d)", head_dim);
        CHECK(rope_dim == 0, "rope_dim must be 0 for the MXFP4 record");
        rec_bytes = head_dim / 2 + head_dim / 32;
    }
    psk_status st = check_cache(cache, num_pages, page_stride, block_size, rec_bytes);
    if (st != PSK_OK) return st;
    CHECK(idx_stride >= cols, "idx_stride must be >= cols");
    if (rows == 0 || cols == 0) return ok();
    CHECK(out != nullptr && indices != nullptr, "out and indices must be non-null");
    CHECK(aligned(out, 16), "out must be 16-byte aligned");
    CHECK(out_stride_t >= 0 && out_stride_j >= 0 && out_stride_t % 8 == 0 &&
              out_stride_j % 8 == 0,
          "output strides must be non-negative multiples of 8 elements");
    CHECK(aligned(indices, 4), "indices must be 4-byte aligned");
    CHECK(rows <= INT64_MAX / (cols > 0 ? cols : 1), "rows * cols overflows");
    psk::GatherParams p{static_cast<uint16_t*>(out), out_stride_t, out_stride_j, cache,
                        num_pages, page_stride, block_size, (int32_t)record, head_dim,
                        rope_dim, is_ue8m0, indices, idx_stride, rows, cols};
    return cuda_status(psk::launch_gather(p, reinterpret_cast<cudaStream_t>(stream)),
                       "dequantize_and_gather_k_cache launch");
}

psk_status dequantize_and_gather_k_cache_ranges(
    void* out, int64_t out_stride_r, int64_t out_stride_i, int64_t out_rows, const uint8_t* cache,
    int64_t num_pages, int64_t page_stride, int32_t block_size, psk_record record,
    int32_t head_dim, int32_t rope_dim, int32_t is_ue8m0, const int32_t* seq_lens,
    const int32_t* gather_lens, const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* base_offsets, int32_t num_reqs, int64_t offset, psk_stream_t stream) {
    if (record != PSK_REC_FP8_DS_MLA)
        return fail(PSK_ERR_UNSUPPORTED, "the range form gathers fp8_ds_mla records only");
    CHECK(is_ue8m0 == 0 || is_ue8m0 == 1, "is_ue8m0 must be 0 or 1");
    CHECK(fp8_head_dim_ok(head_dim), "head_dim must be one of 64, 128, 256, 512, 1024 (got %d)",
          head_dim);
    CHECK(rope_dim >= 0 && rope_dim < head_dim && rope_dim % 64 == 0,
          "rope_dim must be a multiple of 64 in [0, head_dim) (got %d)", rope_dim);
    psk_status st = check_cache(cache, num_pages, page_stride, block_size,
                                fp8_record_bytes(head_dim, rope_dim, is_ue8m0));
    if (st != PSK_OK) return st;
    CHECK(num_reqs >= 0, "num_reqs must be >= 0");
    CHECK(offset >= 0 && out_rows >= offset, "need 0 <= offset <= out_rows");
    CHECK(out_rows - offset <= INT32_MAX, "out_rows - offset must fit in int32");
    CHECK(bt_width >= 0 && bt_stride >= bt_width, "need 0 <= bt_width <= bt_stride");
    if (num_reqs == 0 || out_rows == offset) return ok();
    CHECK(out && seq_lens, "out and seq_lens must be non-null");
    CHECK(bt_width == 0 || block_table, "block_table must be non-null");
    CHECK(aligned(out, 16), "out must be 16-byte aligned");
    CHECK(out_stride_r >= 0 && out_stride_i >= 0 && out_stride_r % 8 == 0 && out_stride_i % 8 == 0,
          "output strides must be non-negative multiples of 8 elements");
    CHECK(aligned(seq_lens, 4) && aligned(gather_lens, 4) && aligned(block_table, 4) &&
              aligned(base_offsets, 4),
          "int32 arrays must be 4-byte aligned");
    psk::RangeParams p{static_cast<uint16_t*>(out), out_stride_r, out_stride_i, out_rows, offset,
                       cache, num_pages, page_stride, block_size, head_dim, rope_dim, is_ue8m0,
                       seq_lens, gather_lens, block_table, bt_stride, bt_width, base_offsets,
                       num_reqs};
    return cuda_status(psk::launch_gather_ranges(p, reinterpret_cast<cudaStream_t>(stream)),
                       "dequantize_and_gather_k_cache_ranges launch");
}

psk_status combine_topk_swa_workspace_indices(
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* gather_lens,
    const int32_t* token_to_req, int32_t num_reqs, int64_t num_tokens, int32_t window,
    int32_t compress_ratio, const int32_t* topk_local, int64_t topk_stride, int32_t topk,
    int64_t workspace_width, int64_t compressed_base, const uint8_t* is_valid_token,
    int32_t* indices, int64_t out_stride, int32_t* lens, psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(window >= 0 && topk >= 0, "window and topk must be >= 0");
    CHECK(compress_ratio >= 1, "compress_ratio must be >= 1");
    CHECK(workspace_width >= 0 && compressed_base >= 0,
          "workspace_width and compressed_base must be >= 0");
    const int64_t cols = (int64_t)window + ((int64_t)topk + 3) / 4 * 4;
    CHECK(cols <= INT32_MAX, "window + padded topk overflows int32");
    CHECK(topk_stride >= topk, "topk_stride must be >= topk");
    CHECK(out_stride >= cols, "out_stride must be >= window + roundup(topk, 4)");
    if (num_tokens == 0) return ok();
    CHECK(num_reqs >= 1, "num_reqs must be >= 1");
    CHECK(query_start_loc && seq_lens && gather_lens && token_to_req && indices && lens,
          "query_start_loc, seq_lens, gather_lens, token_to_req, indices and lens must be non-null");
    CHECK(topk == 0 || topk_local, "topk_local must be non-null");
    CHECK(aligned(query_start_loc, 4) && aligned(seq_lens, 4) && aligned(gather_lens, 4) &&
              aligned(token_to_req, 4) && aligned(topk_local, 4) && aligned(indices, 4) &&
              aligned(lens, 4),
          "int32 arrays must be 4-byte aligned");
    psk::WorkspaceIndexParams p{query_start_loc, seq_lens, gather_lens, token_to_req, num_reqs,
                                num_tokens, window, compress_ratio, topk_local, topk_stride,
                                topk, workspace_width, compressed_base, is_valid_token, indices,
                                out_stride, lens, nullptr};
    return cuda_status(psk::launch_workspace_indices(p, reinterpret_cast<cudaStream_t>(stream)),
                       "combine_topk_swa_workspace_indices launch");
}

psk_status indexer_mxfp4_paged_gather(uint8_t* values_out, uint8_t* scales_out,
                                      const uint8_t* cache, int64_t num_pages,
                                      int64_t page_stride, int32_t block_size, int32_t head_dim,
                                      const int32_t* block_table, int64_t bt_stride,
                                      int32_t bt_width, const int32_t* cu_seq_lens,
                                      int32_t num_reqs, int64_t total_rows,
                                      psk_stream_t stream) {
    CHECK(mxfp4_head_dim_ok(head_dim),
          "head_dim must be one of 32, 64, 128, 256, 512, 1024 (got %d)", head_dim);
    psk_status st = check_cache(cache, num_pages, page_stride, block_size,
                                head_dim / 2 + head_dim / 32);
    if (st != PSK_OK) return st;
    CHECK(total_rows >= 0 && num_reqs >= 0, "total_rows and num_reqs must be >= 0");
    CHECK(bt_width >= 0 && bt_stride >= bt_width, "need 0 <= bt_width <= bt_stride");
    if (total_rows == 0) return ok();
    CHECK(num_reqs >= 1, "num_reqs must be >= 1 when total_rows > 0");
    CHECK(values_out && scales_out && cu_seq_lens, "outputs and cu_seq_lens must be non-null");
    CHECK(bt_width == 0 || block_table, "block_table must be non-null");
    CHECK(aligned(values_out, 4) && aligned(scales_out, 4) && aligned(cu_seq_lens, 4) &&
              aligned(block_table, 4),
          "values_out, scales_out and int32 arrays must be 4-byte aligned");
    psk::RawGatherParams p{values_out, scales_out, cache, num_pages, page_stride, block_size,
                           head_dim, block_table, bt_stride, bt_width, cu_seq_lens, num_reqs,
                           total_rows};
    return cuda_status(psk::launch_mxfp4_raw_gather(p, reinterpret_cast<cudaStream_t>(stream)),
                       "indexer_mxfp4_paged_gather launch");
}

psk_status decode_swa_indices_and_lens(
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* token_to_req,
    int32_t num_reqs, int64_t num_tokens, const int32_t* block_table, int64_t bt_stride,
    int32_t bt_width, const int32_t* base_offsets, int32_t block_size, int32_t window,
    const uint8_t* is_valid_token, int32_t* out_indices, int64_t out_stride, int32_t* out_lens,
    psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(window >= 0, "window must be >= 0");
    CHECK(block_size >= 1, "block_size must be >= 1");
    CHECK(bt_width >= 0 && bt_stride >= bt_width, "need 0 <= bt_width <= bt_stride");
    CHECK(out_stride >= window, "out_stride must be >= window");
    if (num_tokens == 0) return ok();
    CHECK(num_reqs >= 1, "num_reqs must be >= 1");
    CHECK(query_start_loc && seq_lens && token_to_req && out_indices && out_lens,
          "query_start_loc, seq_lens, token_to_req, out_indices and out_lens must be non-null");
    CHECK(bt_width == 0 || block_table, "block_table must be non-null");
    CHECK(aligned(query_start_loc, 4) && aligned(seq_lens, 4) && aligned(token_to_req, 4) &&
              aligned(block_table, 4) && aligned(base_offsets, 4) && aligned(out_indices, 4) &&
              aligned(out_lens, 4),
          "int32 arrays must be 4-byte aligned");
    psk::IndexParams p{};
    p.qsl = query_start_loc;
    p.seq_lens = seq_lens;
    p.t2r = token_to_req;
    p.replay = nullptr;
    p.num_reqs = num_reqs;
    p.num_tokens = num_tokens;
    p.swa_bt = p.comp_bt = block_table;
    p.swa_stride = p.comp_stride = bt_stride;
    p.swa_width = p.comp_width = bt_width;
    p.swa_base = p.comp_base = base_offsets;
    p.swa_bs = p.comp_bs = block_size;
    p.swa_shift = p.comp_shift = psk::log2_if_pow2(block_size);
    p.window = window;
    p.topk = 0;
    p.out_cols = window;
    p.topk_local = nullptr;
    p.topk_stride = 0;
    p.valid = is_valid_token;
    p.out = out_indices;
    p.out_stride = out_stride;
    p.lens = out_lens;
    return cuda_status(psk::launch_index_build(p, true, reinterpret_cast<cudaStream_t>(stream)),
                       "decode_swa_indices_and_lens launch");
}

psk_status compute_dense_compressed_indices_and_lens(
    const int64_t* positions, int64_t num_tokens, const int32_t* token_to_req, int32_t num_reqs,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width, const int32_t* base_offsets,
    int32_t block_size, int32_t compress_ratio, int32_t width, const uint8_t* is_valid_token,
    int32_t* out_indices, int64_t out_stride, int32_t* out_lens, psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(width >= 0, "width must be >= 0");
    CHECK(compress_ratio >= 1, "compress_ratio must be >= 1");
    CHECK(block_size >= 1, "block_size must be >= 1");
    CHECK(bt_width >= 0 && bt_stride >= bt_width, "need 0 <= bt_width <= bt_stride");
    CHECK(out_stride >= width, "out_stride must be >= width");
    if (num_tokens == 0) return ok();
    CHECK(num_reqs >= 1, "num_reqs must be >= 1");
    CHECK(positions && token_to_req && out_lens,
          "positions, token_to_req and out_lens must be non-null");
    CHECK(width == 0 || out_indices, "out_indices must be non-null");
    CHECK(bt_width == 0 || block_table, "block_table must be non-null");
    CHECK(aligned(positions, 8), "positions must be 8-byte aligned");
    CHECK(aligned(token_to_req, 4) && aligned(block_table, 4) && aligned(base_offsets, 4) &&
              aligned(out_indices, 4) && aligned(out_lens, 4),
          "int32 arrays must be 4-byte aligned");
    CHECK(num_tokens <= ((int64_t)INT32_MAX * 256) / (width > 0 ? width : 1),
          "num_tokens x width is too large");
    psk::DenseParams p{positions, num_tokens, token_to_req, num_reqs, block_table, bt_stride,
                       bt_width, base_offsets, block_size, compress_ratio, width, is_valid_token,
                       out_indices, out_stride, out_lens};
    return cuda_status(psk::launch_dense_indices(p, true, reinterpret_cast<cudaStream_t>(stream)),
                       "compute_dense_compressed_indices_and_lens launch");
}

psk_status build_dense_prefill_local_compressed_indices(const int64_t* positions,
                                                        int64_t num_tokens,
                                                        int32_t compress_ratio, int32_t width,
                                                        int32_t* out, int64_t out_stride,
                                                        psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(width >= 0, "width must be >= 0");
    CHECK(compress_ratio >= 1, "compress_ratio must be >= 1");
    CHECK(out_stride >= width, "out_stride must be >= width");
    if (num_tokens == 0 || width == 0) return ok();
    CHECK(positions && out, "positions and out must be non-null");
    CHECK(aligned(positions, 8), "positions must be 8-byte aligned");
    CHECK(aligned(out, 4), "out must be 4-byte aligned");
    CHECK(num_tokens <= ((int64_t)INT32_MAX * 256) / width, "num_tokens x width is too large");
    psk::DenseParams p{};
    p.positions = positions;
    p.num_tokens = num_tokens;
    p.ratio = compress_ratio;
    p.width = width;
    p.bs = 1;
    p.out = out;
    p.out_stride = out_stride;
    return cuda_status(psk::launch_dense_indices(p, false, reinterpret_cast<cudaStream_t>(stream)),
                       "build_dense_prefill_local_compressed_indices launch");
}

psk_status combine_dense_swa_indices(const int64_t* positions, const int32_t* token_to_req,
                                     const int32_t* seq_lens, const int32_t* gather_lens,
                                     int32_t num_reqs, int64_t num_tokens, int32_t window,
                                     int64_t workspace_width, int64_t compressed_base,
                                     int32_t* indices, int64_t out_stride, int32_t* lens,
                                     psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(window >= 0, "window must be >= 0");
    CHECK(workspace_width >= 0 && compressed_base >= 0,
          "workspace_width and compressed_base must be >= 0");
    CHECK(out_stride >= window, "out_stride must be >= window");
    if (num_tokens == 0) return ok();
    CHECK(num_reqs >= 1, "num_reqs must be >= 1");
    CHECK(positions && token_to_req && seq_lens && gather_lens && indices && lens,
          "positions, token_to_req, seq_lens, gather_lens, indices and lens must be non-null");
    CHECK(aligned(positions, 8), "positions must be 8-byte aligned");
    CHECK(aligned(token_to_req, 4) && aligned(seq_lens, 4) && aligned(gather_lens, 4) &&
              aligned(indices, 4) && aligned(lens, 4),
          "int32 arrays must be 4-byte aligned");
    psk::WorkspaceIndexParams p{nullptr, seq_lens, gather_lens, token_to_req, num_reqs,
                                num_tokens, window, 1, nullptr, 0, 0, workspace_width,
                                compressed_base, nullptr, indices, out_stride, lens, positions};
    return cuda_status(psk::launch_workspace_indices(p, reinterpret_cast<cudaStream_t>(stream)),
                       "combine_dense_swa_indices launch");
}

psk_status write_indexer_fp8_cache(const void* index_k, int64_t k_row_stride,
                                   const int64_t* slot_mapping, int64_t num_tokens,
                                   uint8_t* cache, int64_t num_pages, int64_t page_stride,
                                   int32_t block_size, int32_t head_dim, int32_t* err_count,
                                   psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(mxfp4_head_dim_ok(head_dim),
          "head_dim must be one of 32, 64, 128, 256, 512, 1024 (got %d)", head_dim);
    psk_status st = check_cache(cache, num_pages, page_stride, block_size, head_dim + 4);
    if (st != PSK_OK) return st;
    if (num_tokens == 0) return ok();
    CHECK(index_k != nullptr && slot_mapping != nullptr,
          "index_k and slot_mapping must be non-null");
    CHECK(aligned(index_k, 16), "index_k must be 16-byte aligned");
    CHECK(k_row_stride >= head_dim && k_row_stride % 8 == 0,
          "k_row_stride must be >= head_dim and a multiple of 8 elements");
    CHECK(aligned(slot_mapping, 8), "slot_mapping must be 8-byte aligned");
    CHECK(err_count == nullptr || aligned(err_count, 4), "err_count must be 4-byte aligned");
    psk::InsertParams p{index_k, k_row_stride, slot_mapping, num_tokens, cache, num_pages,
                        page_stride, block_size, head_dim, 0, 1, err_count};
    return cuda_status(psk::launch_fp8_indexer_insert(p, reinterpret_cast<cudaStream_t>(stream)),
                       "write_indexer_fp8_cache launch");
}

psk_status indexer_k_norm_rope_store(const void* k_pre, int64_t k_row_stride,
                                     const int64_t* positions, const float* cos_sin_cache,
                                     int64_t cs_stride, int64_t max_pos,
                                     const float* rms_norm_weight, float rms_norm_eps,
                                     const int64_t* kv_slot_mapping, int64_t num_tokens,
                                     int32_t compress_ratio, psk_record record,
                                     uint8_t* k_cache, int64_t num_pages, int64_t page_stride,
                                     int32_t block_size, int32_t* err_count,
                                     psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(record == PSK_REC_MXFP4 || record == PSK_REC_FP8_INDEXER,
          "record must be PSK_REC_MXFP4 or PSK_REC_FP8_INDEXER (got %d)", (int)record);
    CHECK(compress_ratio >= 1, "compress_ratio must be >= 1");
    CHECK(max_pos >= 0 && cs_stride >= 64, "need max_pos >= 0 and cs_stride >= 64");
    psk_status st = check_cache(k_cache, num_pages, page_stride, block_size,
                                record == PSK_REC_MXFP4 ? 68 : 132);
    if (st != PSK_OK) return st;
    if (num_tokens == 0) return ok();
    CHECK(k_pre && positions && cos_sin_cache && rms_norm_weight && kv_slot_mapping,
          "k_pre, positions, cos_sin_cache, rms_norm_weight and kv_slot_mapping must be non-null");
    CHECK(aligned(k_pre, 16) && k_row_stride >= 128 && k_row_stride % 8 == 0,
          "k_pre must be 16-byte aligned with a row stride >= 128 and a multiple of 8 elements");
    CHECK(aligned(positions, 8) && aligned(kv_slot_mapping, 8),
          "positions and kv_slot_mapping must be 8-byte aligned");
    CHECK(aligned(cos_sin_cache, 4), "cos_sin_cache must be 4-byte aligned");
    CHECK(aligned(rms_norm_weight, 16), "rms_norm_weight must be 16-byte aligned");
    CHECK(err_count == nullptr || aligned(err_count, 4), "err_count must be 4-byte aligned");
    CHECK(num_tokens <= INT64_MAX / 32, "num_tokens is too large");
    psk::NormRopeParams p{static_cast<const uint16_t*>(k_pre), k_row_stride, positions,
                          cos_sin_cache, cs_stride, max_pos, rms_norm_weight, rms_norm_eps,
                          kv_slot_mapping, num_tokens, compress_ratio, (int32_t)record, k_cache,
                          num_pages, page_stride, block_size, err_count};
    return cuda_status(psk::launch_norm_rope_store(p, reinterpret_cast<cudaStream_t>(stream)),
                       "indexer_k_norm_rope_store launch");
}

psk_status save_compressor_state(const float* kv, const float* score, int64_t in_stride,
                                 const float* ape, int32_t state_width,
                                 const int64_t* slot_mapping, const int64_t* positions,
                                 int64_t num_tokens, int32_t compress_ratio, float* state_cache,
                                 int64_t num_pages, int32_t block_size, int32_t* err_count,
                                 psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(state_width > 0 && state_width % 4 == 0, "state_width must be a positive multiple of 4");
    CHECK(compress_ratio >= 1, "compress_ratio must be >= 1");
    CHECK(num_pages >= 1 && block_size >= 1, "num_pages and block_size must be >= 1");
    CHECK(state_cache != nullptr && aligned(state_cache, 16), "state_cache must be 16-byte aligned");
    if (num_tokens == 0) return ok();
    CHECK(kv && score && ape && slot_mapping && positions,
          "kv, score, ape, slot_mapping and positions must be non-null");
    CHECK(in_stride >= state_width && in_stride % 4 == 0,
          "in_stride must be >= state_width and a multiple of 4");
    CHECK(aligned(kv, 16) && aligned(score, 16) && aligned(ape, 16),
          "kv, score and ape must be 16-byte aligned");
    CHECK(aligned(slot_mapping, 8) && aligned(positions, 8),
          "slot_mapping and positions must be 8-byte aligned");
    CHECK(err_count == nullptr || aligned(err_count, 4), "err_count must be 4-byte aligned");
    CHECK(num_tokens <= INT64_MAX / 32, "num_tokens is too large");
    psk::SaveStateParams p{kv, score, in_stride, ape, state_width, slot_mapping, positions,
                           num_tokens, compress_ratio, state_cache, num_pages, block_size,
                           err_count};
    return cuda_status(psk::launch_save_compressor_state(p, reinterpret_cast<cudaStream_t>(stream)),
                       "save_compressor_state launch");
}

psk_status compress_kv_cache_insert(
    const float* state_cache, int64_t state_num_pages, int32_t state_block_size,
    int32_t state_width, const int32_t* token_to_req, const int64_t* positions,
    const int64_t* state_slot_mapping, const int32_t* block_table, int64_t bt_stride,
    int32_t bt_width, const int32_t* base_offsets, int32_t num_reqs, int64_t num_tokens,
    int32_t compress_ratio, int32_t overlap, const float* rms_norm_weight, float rms_norm_eps,
    const float* cos_sin_cache, int64_t cs_stride, int64_t max_pos, uint8_t* kv_cache,
    int64_t kv_num_pages, int64_t kv_page_stride, int32_t kv_block_size,
    const int64_t* kv_slot_mapping, int32_t* err_count, psk_stream_t stream) {
    CHECK(num_tokens >= 0, "num_tokens must be >= 0");
    CHECK(overlap == 0 || overlap == 1, "overlap must be 0 or 1");
    CHECK(compress_ratio >= 1 && (overlap ? 2 : 1) * (int64_t)compress_ratio <= 256,
          "the window ((overlap ? 2 : 1) * compress_ratio) must be in [1, 256]");
    CHECK(state_width == (overlap ? 2 : 1) * 512,
          "state_width must be 512 (1024 with overlap) for 512-dim keys");
    CHECK(state_num_pages >= 1 && state_block_size >= 1, "state pages and block size must be >= 1");
    CHECK(bt_width >= 0 && bt_stride >= bt_width, "need 0 <= bt_width <= bt_stride");
    CHECK(max_pos >= 0 && cs_stride >= 64, "need max_pos >= 0 and cs_stride >= 64");
    psk_status st = check_cache(kv_cache, kv_num_pages, kv_page_stride, kv_block_size,
                                fp8_record_bytes(512, 64, 1));
    if (st != PSK_OK) return st;
    if (num_tokens == 0) return ok();
    CHECK(num_reqs >= 1, "num_reqs must be >= 1");
    CHECK(state_cache && token_to_req && positions && state_slot_mapping && rms_norm_weight &&
              cos_sin_cache && kv_slot_mapping,
          "state_cache, token_to_req, positions, state_slot_mapping, rms_norm_weight, "
          "cos_sin_cache and kv_slot_mapping must be non-null");
    CHECK(bt_width == 0 || block_table, "block_table must be non-null");
    CHECK(aligned(state_cache, 16) && aligned(rms_norm_weight, 16),
          "state_cache and rms_norm_weight must be 16-byte aligned");
    CHECK(aligned(positions, 8) && aligned(state_slot_mapping, 8) && aligned(kv_slot_mapping, 8),
          "positions and slot mappings must be 8-byte aligned");
    CHECK(aligned(token_to_req, 4) && aligned(block_table, 4) && aligned(base_offsets, 4) &&
              aligned(cos_sin_cache, 4),
          "int32 arrays and cos_sin_cache must be 4-byte aligned");
    CHECK(err_count == nullptr || aligned(err_count, 4), "err_count must be 4-byte aligned");
    CHECK(num_tokens <= 0x7FFFFFFFll, "num_tokens must fit a grid");
    psk::CompressParams p{state_cache, state_num_pages, state_block_size, state_width,
                          token_to_req, positions, state_slot_mapping, block_table, bt_stride,
                          bt_width, base_offsets, num_reqs, num_tokens, compress_ratio, overlap,
                          rms_norm_weight, rms_norm_eps, cos_sin_cache, cs_stride, max_pos,
                          kv_cache, kv_num_pages, kv_page_stride, kv_block_size, kv_slot_mapping,
                          err_count};
    return cuda_status(psk::launch_compress_kv_insert(p, reinterpret_cast<cudaStream_t>(stream)),
                       "compress_kv_cache_insert launch");
}

psk_status dequantize_and_gather_k_cache_topk(
    void* out, int64_t out_stride_t, int64_t out_stride_j, const uint8_t* cache,
    int64_t num_pages, int64_t page_stride, int32_t block_size, psk_record record,
    int32_t head_dim, int32_t rope_dim, const int32_t* topk_local, int64_t topk_stride,
    int64_t num_tokens, int32_t topk, const int32_t* token_to_req, const int32_t* block_table,
    int64_t bt_stride, int32_t bt_width, int32_t num_reqs, const int32_t* base_offsets,
    const uint8_t* is_valid_token, psk_stream_t stream) {
    CHECK(num_tokens >= 0 && topk >= 0, "num_tokens and topk must be >= 0");
    CHECK(record == PSK_REC_FP8_DS_MLA || record == PSK_REC_MXFP4 ||
              record == PSK_REC_FP8_INDEXER,
          "unknown record %d", (int)record);
    int64_t rec_bytes;
    if (record == PSK_REC_FP8_DS_MLA) {
        CHECK(fp8_head_dim_ok(head_dim),
              "head_dim must be one of 64, 128, 256, 512, 1024 (got %d)", head_dim);
        CHECK(rope_dim >= 0 && rope_dim < head_dim && rope_dim % 64 == 0,
              "rope_dim must be a multiple of 64 in [0, head_dim) (got %d)", rope_dim);
        rec_bytes = fp8_record_bytes(head_dim, rope_dim, 1);
    } else {
        CHECK(mxfp4_head_dim_ok(head_dim),
              "head_dim must be one of 32, 64, 128, 256, 512, 1024 (got %d)", head_dim);
        CHECK(rope_dim == 0, "rope_dim must be 0 for this record");
        rec_bytes = record == PSK_REC_MXFP4 ? head_dim / 2 + head_dim / 32 : head_dim + 4;
    }
    psk_status st = check_cache(cache, num_pages, page_stride, block_size, rec_bytes);
    if (st != PSK_OK) return st;
    CHECK(topk_stride >= topk, "topk_stride must be >= topk");
    CHECK(bt_width >= 0 && bt_stride >= bt_width, "need 0 <= bt_width <= bt_stride");
    if (num_tokens == 0 || topk == 0) return ok();
    CHECK(num_reqs >= 1, "num_reqs must be >= 1");
    CHECK(out && topk_local && token_to_req, "out, topk_local and token_to_req must be non-null");
    CHECK(bt_width == 0 || block_table, "block_table must be non-null");
    CHECK(aligned(out, 16), "out must be 16-byte aligned");
    CHECK(out_stride_t >= 0 && out_stride_j >= 0 && out_stride_t % 8 == 0 && out_stride_j % 8 == 0,
          "output strides must be non-negative multiples of 8 elements");
    CHECK(aligned(topk_local, 4) && aligned(token_to_req, 4) && aligned(block_table, 4) &&
              aligned(base_offsets, 4),
          "int32 arrays must be 4-byte aligned");
    psk::GatherParams p{static_cast<uint16_t*>(out), out_stride_t, out_stride_j, cache,
                        num_pages, page_stride, block_size, (int32_t)record, head_dim,
                        rope_dim, 1, nullptr, 0, num_tokens, topk};
    psk::TopkSource tk{topk_local, topk_stride, token_to_req, is_valid_token, num_reqs,
                       block_table, bt_stride, bt_width, base_offsets};
    return cuda_status(psk::launch_gather_topk(p, tk, reinterpret_cast<cudaStream_t>(stream)),
                       "dequantize_and_gather_k_cache_topk launch");
}

psk_status dequantize_and_gather_k_cache_window(
    void* out, int64_t out_stride_t, int64_t out_stride_j, const uint8_t* cache,
    int64_t num_pages, int64_t page_stride, int32_t block_size, int32_t head_dim,
    int32_t rope_dim, const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* token_to_req, const int32_t* replay_start, int32_t num_reqs,
    int64_t num_tokens, const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* base_offsets, int32_t window, const uint8_t* is_valid_token,
    psk_stream_t stream) {
    CHECK(num_tokens >= 0 && window >= 0, "num_tokens and window must be >= 0");
    CHECK(fp8_head_dim_ok(head_dim),
          "head_dim must be one of 64, 128, 256, 512, 1024 (got %d)", head_dim);
    CHECK(rope_dim >= 0 && rope_dim < head_dim && rope_dim % 64 == 0,
          "rope_dim must be a multiple of 64 in [0, head_dim) (got %d)", rope_dim);
    psk_status st = check_cache(cache, num_pages, page_stride, block_size,
                                fp8_record_bytes(head_dim, rope_dim, 1));
    if (st != PSK_OK) return st;
    CHECK(bt_width >= 0 && bt_stride >= bt_width, "need 0 <= bt_width <= bt_stride");
    if (num_tokens == 0 || window == 0) return ok();
    CHECK(num_reqs >= 1, "num_reqs must be >= 1");
    CHECK(out && query_start_loc && seq_lens && token_to_req,
          "out, query_start_loc, seq_lens and token_to_req must be non-null");
    CHECK(bt_width == 0 || block_table, "block_table must be non-null");
    CHECK(aligned(out, 16), "out must be 16-byte aligned");
    CHECK(out_stride_t >= 0 && out_stride_j >= 0 && out_stride_t % 8 == 0 && out_stride_j % 8 == 0,
          "output strides must be non-negative multiples of 8 elements");
    CHECK(aligned(query_start_loc, 4) && aligned(seq_lens, 4) && aligned(token_to_req, 4) &&
              aligned(replay_start, 4) && aligned(block_table, 4) && aligned(base_offsets, 4),
          "int32 arrays must be 4-byte aligned");
    psk::GatherParams p{static_cast<uint16_t*>(out), out_stride_t, out_stride_j, cache,
                        num_pages, page_stride, block_size, 0, head_dim, rope_dim, 1, nullptr, 0,
                        num_tokens, window};
    psk::WindowSource wn{query_start_loc, seq_lens, token_to_req, replay_start, is_valid_token,
                         num_reqs, block_table, bt_stride, bt_width, base_offsets};
    return cuda_status(psk::launch_gather_window(p, wn, reinterpret_cast<cudaStream_t>(stream)),
                       "dequantize_and_gather_k_cache_window launch");
}

psk_status dequantize_and_gather_k_cache_pair(
    void* out, int64_t out_stride_t, int64_t out_stride_j, const uint8_t* cache_a,
    int64_t num_pages_a, int64_t page_stride_a, int32_t block_size_a, const uint8_t* cache_b,
    int64_t num_pages_b, int64_t page_stride_b, int32_t block_size_b, int32_t head_dim,
    int32_t rope_dim, const int32_t* indices, int64_t idx_stride, int64_t rows, int32_t cols,
    int32_t split, psk_stream_t stream) {
    CHECK(rows >= 0 && cols >= 0, "rows and cols must be >= 0");
    CHECK(split >= 0 && split <= cols, "need 0 <= split <= cols");
    CHECK(fp8_head_dim_ok(head_dim),
          "head_dim must be one of 64, 128, 256, 512, 1024 (got %d)", head_dim);
    CHECK(rope_dim >= 0 && rope_dim < head_dim && rope_dim % 64 == 0,
          "rope_dim must be a multiple of 64 in [0, head_dim) (got %d)", rope_dim);
    const int64_t rec_bytes = fp8_record_bytes(head_dim, rope_dim, 1);
    psk_status st = check_cache(cache_a, num_pages_a, page_stride_a, block_size_a, rec_bytes);
    if (st != PSK_OK) return st;
    st = check_cache(cache_b, num_pages_b, page_stride_b, block_size_b, rec_bytes);
    if (st != PSK_OK) return st;
    CHECK(idx_stride >= cols, "idx_stride must be >= cols");
    if (rows == 0 || cols == 0) return ok();
    CHECK(out != nullptr && indices != nullptr, "out and indices must be non-null");
    CHECK(aligned(out, 16), "out must be 16-byte aligned");
    CHECK(out_stride_t >= 0 && out_stride_j >= 0 && out_stride_t % 8 == 0 &&
              out_stride_j % 8 == 0,
          "output strides must be non-negative multiples of 8 elements");
    CHECK(aligned(indices, 4), "indices must be 4-byte aligned");
    CHECK(rows <= INT64_MAX / cols, "rows * cols overflows");
    psk::GatherParams p{static_cast<uint16_t*>(out), out_stride_t, out_stride_j, cache_a,
                        num_pages_a, page_stride_a, block_size_a, 0, head_dim, rope_dim, 1,
                        indices, idx_stride, rows, cols};
    psk::PairSource pr{cache_b, num_pages_b, page_stride_b, block_size_b, -1, split};
    return cuda_status(psk::launch_gather_pair(p, pr, reinterpret_cast<cudaStream_t>(stream)),
                       "dequantize_and_gather_k_cache_pair launch");
}

psk_status dequantize_and_gather_k_cache_dense(
    void* out, int64_t out_stride_t, int64_t out_stride_j, const uint8_t* cache,
    int64_t num_pages, int64_t page_stride, int32_t block_size, int32_t head_dim,
    int32_t rope_dim, const int64_t* positions, int64_t num_tokens, const int32_t* token_to_req,
    int32_t num_reqs, const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* base_offsets, int32_t compress_ratio, int32_t width,
    const uint8_t* is_valid_token, psk_stream_t stream) {
    CHECK(num_tokens >= 0 && width >= 0, "num_tokens and width must be >= 0");
    CHECK(compress_ratio >= 1, "compress_ratio must be >= 1");
    CHECK(fp8_head_dim_ok(head_dim),
          "head_dim must be one of 64, 128, 256, 512, 1024 (got %d)", head_dim);
    CHECK(rope_dim >= 0 && rope_dim < head_dim && rope_dim % 64 == 0,
          "rope_dim must be a multiple of 64 in [0, head_dim) (got %d)", rope_dim);
    psk_status st = check_cache(cache, num_pages, page_stride, block_size,
                                fp8_record_bytes(head_dim, rope_dim, 1));
    if (st != PSK_OK) return st;
    CHECK(bt_width >= 0 && bt_stride >= bt_width, "need 0 <= bt_width <= bt_stride");
    if (num_tokens == 0 || width == 0) return ok();
    CHECK(num_reqs >= 1, "num_reqs must be >= 1");
    CHECK(out && positions && token_to_req, "out, positions and token_to_req must be non-null");
    CHECK(bt_width == 0 || block_table, "block_table must be non-null");
    CHECK(aligned(out, 16), "out must be 16-byte aligned");
    CHECK(out_stride_t >= 0 && out_stride_j >= 0 && out_stride_t % 8 == 0 && out_stride_j % 8 == 0,
          "output strides must be non-negative multiples of 8 elements");
    CHECK(aligned(positions, 8), "positions must be 8-byte aligned");
    CHECK(aligned(token_to_req, 4) && aligned(block_table, 4) && aligned(base_offsets, 4),
          "int32 arrays must be 4-byte aligned");
    CHECK(num_tokens <= INT64_MAX / width, "num_tokens * width overflows");
    psk::GatherParams p{static_cast<uint16_t*>(out), out_stride_t, out_stride_j, cache,
                        num_pages, page_stride, block_size, 0, head_dim, rope_dim, 1, nullptr, 0,
                        num_tokens, width};
    psk::DenseSource ds{positions, token_to_req, is_valid_token, num_reqs, block_table, bt_stride,
                        bt_width, base_offsets, compress_ratio};
    return cuda_status(psk::launch_gather_dense(p, ds, reinterpret_cast<cudaStream_t>(stream)),
                       "dequantize_and_gather_k_cache_dense launch");
}

}  // extern "C"

namespace psk {

int sm_count() {
    static std::atomic<int> cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace psk
