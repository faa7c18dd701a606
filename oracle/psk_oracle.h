/*
 * psk_oracle.h -- declarations of the CPU oracle for the paged sparse K-cache
 * pipeline.
 *
 * TEST INFRASTRUCTURE ONLY.  This oracle is a plain, slow, single-threaded C
 * restatement of what the pipeline computes.  It exists so that tests, the
 * smoke check and the CPU-baseline leg of the benchmark can check the CUDA
 * path.  Nothing in the product library includes, links or calls it, and it
 * includes nothing from the product library.
 *
 * Parity pins: every function below is pinned by the CPU test-suite against
 * something other than itself (format definitions enumerated exhaustively, a
 * library cast, brute-force enumeration of windows and slots, hand-worked
 * golden records, invariants).  The fp32-scale FP8 record (is_ue8m0 = 0),
 * whose rule no page prints, is pinned by a hand-worked record (insert and
 * gather) and by torch's e4m3 encode and decode.  indexer_k_norm_rope_store takes
 * two readings (pairwise summation, IEEE binary32 square root then division) that fix
 * the rounding of steps the pages leave open; its pins check the arithmetic
 * against closed forms, not a printed result.
 */
#ifndef PSK_ORACLE_H
#define PSK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- scalar formats (OCP OFP8 E4M3FN, OCP MX v1.0 E2M1 / E8M0, bf16) ---- */
uint8_t  oracle_e4m3_encode(float v);
float    oracle_e4m3_decode(uint8_t code);
uint8_t  oracle_e2m1_encode(float v);
float    oracle_e2m1_decode(uint8_t nibble);
int32_t  oracle_ceil_log2(float q);
uint16_t oracle_bf16_from_f32(float f);
float    oracle_bf16_to_f32(uint16_t b);

void oracle_e4m3_encode_array(const float* v, uint8_t* out, int64_t n);
void oracle_e2m1_encode_array(const float* v, uint8_t* out, int64_t n);
void oracle_ceil_log2_array(const float* q, int32_t* out, int64_t n);

/* ---- record geometry ---- */
int64_t oracle_fp8_token_stride(int32_t head_dim, int32_t rope_dim);
int64_t oracle_fp8_scale_bytes(int32_t head_dim, int32_t is_ue8m0);

/* ---- pipeline steps ---- */
int64_t oracle_quantize_and_insert_k_cache(
    const uint16_t* k, int64_t k_row_stride, const int64_t* slot_mapping,
    int64_t num_tokens, uint8_t* cache, int64_t num_pages,
    int64_t page_stride, int32_t block_size, int32_t head_dim,
    int32_t rope_dim, int32_t is_ue8m0);

int64_t oracle_write_indexer_mxfp4_cache(
    const uint16_t* k, int64_t k_row_stride, const int64_t* slot_mapping,
    int64_t num_tokens, uint8_t* cache, int64_t num_pages,
    int64_t page_stride, int32_t block_size, int32_t head_dim);

void oracle_compute_global_topk_indices_and_lens(
    const int32_t* topk_local, int64_t topk_stride, int64_t num_tokens,
    int32_t topk, const int32_t* token_to_req, const int32_t* block_table,
    int64_t bt_stride, int32_t bt_width, int32_t num_reqs, int32_t block_size,
    const int32_t* base_offsets, const uint8_t* is_valid_token,
    int32_t* out_indices, int64_t out_stride, int32_t* out_lens);

void oracle_combine_topk_swa_indices(
    const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* token_to_req, const int32_t* replay_start, int32_t num_reqs,
    int64_t num_tokens,
    const int32_t* swa_block_table, int64_t swa_bt_stride, int32_t swa_bt_width,
    const int32_t* swa_base_offsets, int32_t swa_block_size,
    const int32_t* comp_block_table, int64_t comp_bt_stride,
    int32_t comp_bt_width, const int32_t* comp_base_offsets,
    int32_t comp_block_size, int32_t window, int32_t compress_ratio,
    const int32_t* topk_local, int64_t topk_stride, int32_t topk,
    const uint8_t* is_valid_token, int32_t* sparse_indices, int64_t out_stride,
    int32_t* lens);

void oracle_dequantize_and_gather_k_cache(
    uint16_t* out, int64_t out_stride_t, int64_t out_stride_j,
    const uint8_t* cache, int64_t num_pages, int64_t page_stride,
    int32_t block_size, int32_t record, int32_t head_dim, int32_t rope_dim,
    int32_t is_ue8m0, const int32_t* indices, int64_t idx_stride, int64_t rows,
    int32_t cols);

/* ---- range-form gather, workspace indices, raw MXFP4 gather ---- */
void oracle_dequantize_and_gather_k_cache_ranges(
    uint16_t* out, int64_t out_stride_r, int64_t out_stride_i, int64_t out_rows,
    const uint8_t* cache, int64_t num_pages, int64_t page_stride,
    int32_t block_size, int32_t record, int32_t head_dim, int32_t rope_dim,
    int32_t is_ue8m0, const int32_t* seq_lens, const int32_t* gather_lens,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* base_offsets, int32_t num_reqs, int64_t offset);

void oracle_combine_topk_swa_workspace_indices(
    const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* gather_lens, const int32_t* token_to_req, int32_t num_reqs,
    int64_t num_tokens, int32_t window, int32_t compress_ratio,
    const int32_t* topk_local, int64_t topk_stride, int32_t topk,
    int64_t workspace_width, int64_t compressed_base,
    const uint8_t* is_valid_token, int32_t* indices, int64_t out_stride,
    int32_t* lens);

void oracle_indexer_mxfp4_paged_gather(
    uint8_t* values_out, uint8_t* scales_out, const uint8_t* cache,
    int64_t num_pages, int64_t page_stride, int32_t block_size,
    int32_t head_dim, const int32_t* block_table, int64_t bt_stride,
    int32_t bt_width, const int32_t* cu_seq_lens, int32_t num_reqs);

/* ---- dense builders ---- */
void oracle_decode_swa_indices_and_lens(
    const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* token_to_req, int32_t num_reqs, int64_t num_tokens,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* base_offsets, int32_t block_size, int32_t window,
    const uint8_t* is_valid_token, int32_t* indices, int64_t out_stride,
    int32_t* lens);

void oracle_compute_dense_compressed_indices_and_lens(
    const int64_t* positions, int64_t num_tokens, const int32_t* token_to_req,
    int32_t num_reqs, const int32_t* block_table, int64_t bt_stride,
    int32_t bt_width, const int32_t* base_offsets, int32_t block_size,
    int32_t compress_ratio, int32_t width, const uint8_t* is_valid_token,
    int32_t* indices, int64_t out_stride, int32_t* lens);

void oracle_build_dense_prefill_local_compressed_indices(
    const int64_t* positions, int64_t num_tokens, int32_t compress_ratio,
    int32_t width, int32_t* out, int64_t out_stride);

void oracle_combine_dense_swa_indices(
    const int64_t* positions, const int32_t* token_to_req,
    const int32_t* seq_lens, const int32_t* gather_lens, int32_t num_reqs,
    int64_t num_tokens, int32_t window, int64_t workspace_width,
    int64_t compressed_base, int32_t* indices, int64_t out_stride,
    int32_t* lens);

/* ---- indexer-key variants ---- */
int64_t oracle_write_indexer_fp8_cache(
    const uint16_t* k, int64_t k_row_stride, const int64_t* slot_mapping,
    int64_t num_tokens, uint8_t* cache, int64_t num_pages,
    int64_t page_stride, int32_t block_size, int32_t head_dim);

int64_t oracle_indexer_k_norm_rope_store(
    const uint16_t* k_pre, int64_t k_row_stride, const int64_t* positions,
    const float* cos_sin_cache, int64_t cs_stride, int64_t max_pos,
    const float* rms_norm_weight, float rms_norm_eps,
    const int64_t* slot_mapping, int64_t num_tokens, int32_t compress_ratio,
    int32_t record, uint8_t* cache, int64_t num_pages, int64_t page_stride,
    int32_t block_size);

/* ---- compressed-KV producer ---- */
float oracle_exp_cw(float x);
void oracle_exp_cw_array(const float* x, float* out, int64_t n);

int64_t oracle_save_compressor_state(
    const float* kv, const float* score, int64_t in_stride, const float* ape,
    int32_t state_width, const int64_t* slot_mapping, const int64_t* positions,
    int64_t num_tokens, int32_t compress_ratio, float* state_cache, int64_t num_pages,
    int32_t block_size);

int64_t oracle_compress_kv_cache_insert(
    const float* state_cache, int64_t state_num_pages, int32_t state_block_size,
    int32_t state_width, const int32_t* token_to_req, const int64_t* positions,
    const int64_t* state_slot_mapping, const int32_t* block_table, int64_t bt_stride,
    int32_t bt_width, const int32_t* base_offsets, int32_t num_reqs, int64_t num_tokens,
    int32_t compress_ratio, int32_t overlap, int32_t head_dim, int32_t rope_dim,
    const float* rms_norm_weight, float rms_norm_eps, const float* cos_sin_cache,
    int64_t cs_stride, int64_t max_pos, uint8_t* kv_cache, int64_t kv_num_pages,
    int64_t kv_page_stride, int32_t kv_block_size, const int64_t* kv_slot_mapping);

#ifdef __cplusplus
}
#endif

#endif /* PSK_ORACLE_H */
