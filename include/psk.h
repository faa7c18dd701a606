/*
 * psk.h -- C ABI of libpsk, the GB300 (sm_103a) paged sparse K-cache library.
 *
 * The library implements the hot path of a DeepSeek-V4-style sparse-MLA
 * serving runtime's paged K cache, as stated on these pages:
 *   [OPS]  TokenSpeed runtime/layers/attention/deepseek_v4_ops.py
 *   [BE]   TokenSpeed runtime/layers/attention/backends/deepseek_v4.py
 *   [MDL]  TokenSpeed runtime/models/deepseek_v4.py
 *   [VLLM] vLLM API docs, vllm.models.deepseek_v41.common.ops
 * and the OCP OFP8 (E4M3) and OCP MX v1.0 (E2M1, E8M0) format definitions.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * - Every pointer argument is DEVICE memory owned by the caller.  The library
 *   allocates nothing, keeps no state between calls, never synchronises, and
 *   launches only on `stream` (NULL = the legacy default stream), so calls can
 *   be captured into CUDA graphs.
 * - Strides are in ELEMENTS of the pointed-to type unless the name ends in
 *   `_bytes`/`page_stride`.
 * - bf16 tensors are passed as `void*` pointing at IEEE bfloat16 values.
 * - Argument errors (null required pointer, negative or inconsistent sizes,
 *   unsupported head_dim/rope_dim, misaligned pointer or stride) return
 *   PSK_ERR_INVALID_ARGUMENT before any launch; nothing is written.
 * - Zero work (no tokens, no rows) returns PSK_OK without a launch.
 * - A failed launch returns PSK_ERR_CUDA.
 * - psk_last_error() returns a message for the calling thread's last error.
 * - Data-dependent problems never fault: a slot, page or index outside the
 *   cache or table is skipped or emitted as -1 ("fail closed", [MDL]
 *   _deepseek_v4_swa_slot_mapping), as each entry point states.
 * - Every kernel is launched with programmatic dependent launch: it may start
 *   while the previous kernel on `stream` is finishing, and waits for that
 *   kernel to complete (griddepcontrol.wait, after which its writes are
 *   visible) before it reads any global memory, so every input may be
 *   written by the kernel just before it on the stream.
 *
 * Cache records ("pages")
 * -----------------------
 * A cache is `num_pages` pages of `page_stride` bytes; `block_size` token slots
 * per page; slot s lives in page s / block_size at offset s % block_size.
 *
 * fp8_ds_mla record ([OPS] dequantize_deepseek_v4_fp8_ds_mla_cache,
 * _fp8_ds_mla_cache_rows; [VLLM] quantize_and_insert_k_cache):
 *   nope = head_dim - rope_dim, token_stride = nope + 2 * rope_dim.
 *   page = [block_size x token_stride data][block_size x scale_bytes scales]
 *   data  = nope E4M3 bytes, then rope_dim bf16 values (little-endian).
 *   scales, is_ue8m0 = 1: head_dim/64 bytes, byte b = UE8M0 exponent of 64-block
 *           b (value 2^(byte-127)); slots past the nope blocks are 0.  For
 *           head_dim 512 / rope 64 that is 7 scales + 1 zero pad = 8 bytes and
 *           the record is 584 bytes.
 *   scales, is_ue8m0 = 0: head_dim/64 little-endian binary32 scales (4 bytes
 *           each); slots past the nope blocks are 0.0.
 *   page_stride >= block_size * (token_stride + scale_bytes).
 *
 * MXFP4 record ([OPS] write/read_deepseek_v4_indexer_mxfp4_cache):
 *   page = [block_size x head_dim/2 value bytes][block_size x head_dim/32 scales]
 *   value byte j holds element 2j in its low nibble, 2j+1 in its high nibble
 *   (E2M1); scale byte b = E8M0 exponent of 32-block b.  68 bytes for 128 dims.
 *
 * Alignment required by the kernels (checked): cache base and page_stride
 * multiples of 16 bytes; bf16 inputs/outputs 16-byte aligned with strides that
 * are multiples of 8 elements; int32 index matrices 4-byte aligned.
 */
#ifndef PSK_H
#define PSK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Identical to cudaStream_t; declared here so callers need no CUDA headers. */
typedef struct CUstream_st* psk_stream_t;

typedef enum psk_status {
    PSK_OK = 0,
    PSK_ERR_INVALID_ARGUMENT = 1,
    PSK_ERR_UNSUPPORTED = 2,
    PSK_ERR_CUDA = 3
} psk_status;

typedef enum psk_record {
    PSK_REC_FP8_DS_MLA = 0,
    PSK_REC_MXFP4 = 1,
    PSK_REC_FP8_INDEXER = 2
} psk_record;

/* Message describing the calling thread's most recent error ("" if none). */
const char* psk_last_error(void);

/* ABI revision of this header (bumped on any signature change). */
int32_t psk_abi_version(void);

/*
 * psk_device_wait_timeouts -- diagnostic of the pipelined kernels.
 * Kernels that wait on shared-memory barriers (the TMA-fed gather, the
 * index builders that stage top-k rows by bulk copies and the long-window
 * compressed-row kernel of compress_kv_cache_insert) bound every wait to
 * 2 s of wall time; a wait that expires is counted in a per-device counter,
 * the kernel stops its remaining work instead of hanging, and the output of
 * that launch is incomplete.  This call copies the current device's count
 * (the sum over those kernels; 0 in normal operation) into *count.  Synchronous (it waits for the
 * device); returns PSK_ERR_CUDA if the copy fails.
 * Once the count has risen, treat every output written on the device since
 * the last check as invalid: the launch that gave up left rows unwritten, and
 * a CTA whose final drain also expired may have retired with bulk copies
 * still landing in its shared memory, which a CTA of a launch running beside
 * it could then be using.
 */
psk_status psk_device_wait_timeouts(uint32_t* count);

/*
 * psk_device_wait_selftest -- exercises the failure path of those bounded
 * waits (the pages have no counterpart; a diagnostic of this library).  One
 * thread of a one-warp kernel waits on a shared-memory barrier that nothing
 * completes; after limit_ns (1e3 .. 1e9 ns) of wall time the wait gives up,
 * the expiry is counted as in the pipelined kernels (psk_device_wait_timeouts
 * rises by one when the kernel has run) and the kernel returns normally, so the
 * context and the stream stay usable.  Asynchronous on `stream`.  Errors:
 * PSK_ERR_INVALID_ARGUMENT for a limit outside the range, PSK_ERR_CUDA if the
 * launch fails.
 */
psk_status psk_device_wait_selftest(uint64_t limit_ns, psk_stream_t stream);

/*
 * quantize_and_insert_k_cache -- block-scaled FP8 quantize + paged insert.
 * [VLLM] quantize_and_insert_k_cache; math of [OPS] _fp8_ds_mla_cache_rows.
 *
 *   k            bf16 [num_tokens, >= head_dim], row stride k_row_stride
 *                (elements, multiple of 8).  Only the first num_tokens rows are
 *                read: num_tokens is the length of slot_mapping, and k may have
 *                more (data-parallel padding) rows.
 *   slot_mapping int64 [num_tokens]; -1 (any negative) = skip the token.
 *   k_cache      uint8 [num_pages, page_stride] fp8_ds_mla pages (written).
 *   head_dim     one of 64, 128, 256, 512, 1024; rope_dim multiple of 64 in
 *                [0, head_dim); the rope dims are the last rope_dim of each row
 *                and are stored verbatim (the caller has already rotated them).
 *   is_ue8m0     1: per 64-block e = ceil(log2(max(amax, 1e-4) / 448)) exactly,
 *                   scale byte e + 127, codes RNE-E4M3(clamp(x * 2^-e, +-448)).
 *                0: scale = max(amax, 1e-12) / 448 (binary32, stored as fp32),
 *                   codes RNE-E4M3(clamp(x / scale, +-448)) with IEEE division.
 *   err_count    nullable device int32: incremented (atomically) once per token
 *                whose slot is >= num_pages * block_size; such tokens are
 *                skipped.  The caller zeroes it when it wants a fresh count.
 */
psk_status quantize_and_insert_k_cache(
    const void* k, int64_t k_row_stride, const int64_t* slot_mapping,
    int64_t num_tokens, uint8_t* k_cache, int64_t num_pages,
    int64_t page_stride, int32_t block_size, int32_t head_dim,
    int32_t rope_dim, int32_t is_ue8m0, int32_t* err_count,
    psk_stream_t stream);

/*
 * write_indexer_mxfp4_cache -- MXFP4 quantize + paged insert of indexer keys.
 * [OPS] write_deepseek_v4_indexer_mxfp4_cache (layout) and
 * read_deepseek_v4_indexer_mxfp4_cache (nibble order, scale meaning).
 *
 *   index_k      bf16 [num_tokens, >= head_dim], row stride k_row_stride.
 *   slot_mapping int64 [num_tokens]; negative = skip.
 *   cache        uint8 [num_pages, page_stride] MXFP4 pages (written).
 *   head_dim     one of 32, 64, 128, 256, 512, 1024.
 *   Per 32-block: e = ceil(log2(max(amax, 1e-4) / 6)) (the pages print no
 *   writer rule; this is E8M0 = ceil-pow2(amax / 6)), scale byte
 *   clamp(e + 127, 0, 254), codes RNE-E2M1 of x * 2^-e, saturating at 6.
 *   err_count    as for quantize_and_insert_k_cache.
 */
psk_status write_indexer_mxfp4_cache(
    const void* index_k, int64_t k_row_stride, const int64_t* slot_mapping,
    int64_t num_tokens, uint8_t* cache, int64_t num_pages,
    int64_t page_stride, int32_t block_size, int32_t head_dim,
    int32_t* err_count, psk_stream_t stream);

/*
 * compute_global_topk_indices_and_lens -- local top-k -> global cache slots.
 * [VLLM] compute_global_topk_indices_and_lens; called for decode in [BE]
 * _decode_compressed_attention_indices_and_lens.
 *
 *   topk_local     int32 [num_tokens, topk], row stride topk_stride; -1 = none.
 *   token_to_req   int32 [num_tokens] request of each token.
 *   block_table    int32 [num_reqs, >= bt_width], row stride bt_stride; -1 = no
 *                  page.
 *   base_offsets   nullable int32 [num_reqs]: logical page of each row's first
 *                  entry (0 when null).
 *   is_valid_token nullable uint8 [num_tokens]: 0 marks a padding token.
 *   out_indices    int32 [num_tokens, topk], row stride out_stride (written):
 *                  out[t][j] = page * block_size + l % block_size with
 *                  l = topk_local[t][j], page = block_table[r][l/block_size - base];
 *                  -1 when l < 0, the logical page is outside [0, bt_width),
 *                  the page is < 0, or the slot exceeds INT32_MAX.  Entries are
 *                  not compacted.
 *   out_lens       int32 [num_tokens]: number of entries >= 0 (0 for a padding
 *                  token, whose entries are all -1; a token whose request index
 *                  is outside [0, num_reqs) is treated as padding).
 */
psk_status compute_global_topk_indices_and_lens(
    const int32_t* topk_local, int64_t topk_stride, int64_t num_tokens,
    int32_t topk, const int32_t* token_to_req, const int32_t* block_table,
    int64_t bt_stride, int32_t bt_width, int32_t num_reqs, int32_t block_size,
    const int32_t* base_offsets, const uint8_t* is_valid_token,
    int32_t* out_indices, int64_t out_stride, int32_t* out_lens,
    psk_stream_t stream);

/*
 * combine_topk_swa_indices -- the fused sparse-index build.
 * [VLLM] build_flashinfer_mixed_sparse_indices (single kernel for a
 * decode-first batch); TokenSpeed calls the same step combine_topk_swa_indices.
 *
 *   query_start_loc int32 [num_reqs + 1]; seq_lens int32 [num_reqs];
 *   token_to_req    int32 [num_tokens]; replay_start nullable int32 [num_reqs]
 *                   (0 when null).  Token t of request r sits at
 *                   pos = seq_lens[r] - (qsl[r+1] - qsl[r]) + (t - qsl[r])
 *                   ([BE] _decode_positions_from_metadata).
 *   swa_*           the sliding-window cache's block table (see
 *                   compute_global_topk_indices_and_lens for the table/base
 *                   convention) and page size.
 *   comp_*          the compressed cache's block table; comp_block_table NULL
 *                   means the SWA table (with its stride and width) is used.
 *                   comp_base_offsets is independent of the table choice.
 *   window          W >= 0; compress_ratio >= 1 (accepted for the signature;
 *                   it does not change the result).
 *   topk_local      int32 [num_tokens, topk], row stride topk_stride.
 *   sparse_indices  int32 [num_tokens, window + roundup(topk, 4)], row stride
 *                   out_stride (written):
 *                   columns [0, W): slots of positions lo, lo+1, ..., pos with
 *                     lo = max(replay_start[r], pos - W + 1, 0), left-aligned
 *                     (oldest first), -1 after pos or where no page exists;
 *                   columns [W, W + topk): top-k mapped through the compressed
 *                     table exactly as compute_global_topk_indices_and_lens;
 *                   remaining columns: -1 (rows start on 16-byte boundaries
 *                     when out_stride is a multiple of 4).
 *   lens            int32 [num_tokens]: entries >= 0 over all columns.
 *   A padding token (is_valid_token 0 or request out of range): all -1, lens 0.
 */
psk_status combine_topk_swa_indices(
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
    int32_t* lens, psk_stream_t stream);

/*
 * dequantize_and_gather_k_cache -- index-keyed dequantize + gather.
 * Index form of [VLLM] dequantize_and_gather_k_cache; per-row math of [OPS]
 * dequantize_deepseek_v4_fp8_ds_mla_cache (record 0),
 * read_deepseek_v4_indexer_mxfp4_cache (record 1) and the FP8 indexer record
 * of write_deepseek_v4_indexer_fp8_cache (record 2).
 *
 *   out          bf16; row (t, j) starts at out + t*out_stride_t + j*out_stride_j
 *                (elements, multiples of 8) and holds head_dim values.
 *   cache        uint8 [num_pages, page_stride] pages of the given record.
 *   indices      int32 [rows, cols], row stride idx_stride: slot ids.
 *   For s = indices[t][j]: s < 0 or s >= num_pages * block_size gives an
 *   all-zero row.  Otherwise, fp8_ds_mla: nope dim d = bf16(e4m3 * 2^(scale-127))
 *   (or * fp32 scale when is_ue8m0 = 0), rope dims copied bit for bit; MXFP4:
 *   dim d = bf16(e2m1 * 2^(scale-127)); FP8 indexer: dim d = bf16(e4m3 *
 *   scale_f32).  Products are formed in binary32 and rounded to bf16 (for
 *   power-of-two scales the product is exact).  MXFP4 and FP8 indexer records
 *   take head_dim in {32, 64, ..., 1024} and rope_dim 0.
 *   To gather the window columns from the SWA cache and the top-k columns from
 *   the compressed cache, make two calls on column ranges of one index matrix
 *   and one output (pointer offsets + strides), as a k_cache / extra_k_cache
 *   pair is read ([BE] forward_deepseek_v4_decode).
 */
psk_status dequantize_and_gather_k_cache(
    void* out, int64_t out_stride_t, int64_t out_stride_j,
    const uint8_t* cache, int64_t num_pages, int64_t page_stride,
    int32_t block_size, psk_record record, int32_t head_dim, int32_t rope_dim,
    int32_t is_ue8m0, const int32_t* indices, int64_t idx_stride, int64_t rows,
    int32_t cols, psk_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Prefill workspace path (TokenSpeed backends/deepseek_v4.py, _prefill_workspace) */
/* ------------------------------------------------------------------------ */

/*
 * dequantize_and_gather_k_cache_ranges -- range-form dequantize + gather.
 * [VLLM] dequantize_and_gather_k_cache(out, k_cache, seq_lens, gather_lens,
 * block_table, block_size, offset); [BE] _prefill_workspace calls it for the
 * compressed cache (offset 0, gather_lens NULL) and the SWA cache (offset
 * compressed_base, gather_lens = query_lens + min(prefix, W - 1)).
 *
 *   out          bf16 [num_reqs, out_rows, head_dim]; row i of request r starts
 *                at out + r*out_stride_r + i*out_stride_i (elements, multiples
 *                of 8).
 *   For request r, g = gather_lens[r] (seq_lens[r] when gather_lens is NULL):
 *   row i in [0, g) is position seq_lens[r] - g + i, mapped through
 *   block_table[r] (logical page position/block_size - base_offsets[r]) and
 *   written, dequantized as dequantize_and_gather_k_cache does, to out row
 *   offset + i; a position without a page gives a zero row.  Rows at or beyond
 *   out_rows, and rows of out outside [offset, offset + g), are not written.
 *   record must be PSK_REC_FP8_DS_MLA (PSK_ERR_UNSUPPORTED otherwise).
 *   Requires 0 <= offset <= out_rows and out_rows - offset <= INT32_MAX.
 */
psk_status dequantize_and_gather_k_cache_ranges(
    void* out, int64_t out_stride_r, int64_t out_stride_i, int64_t out_rows,
    const uint8_t* cache, int64_t num_pages, int64_t page_stride,
    int32_t block_size, psk_record record, int32_t head_dim, int32_t rope_dim,
    int32_t is_ue8m0, const int32_t* seq_lens, const int32_t* gather_lens,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* base_offsets, int32_t num_reqs, int64_t offset,
    psk_stream_t stream);

/*
 * combine_topk_swa_workspace_indices -- workspace-relative fused index build.
 * TokenSpeed's combine_topk_swa_indices(topk_indices, query_start_loc,
 * seq_lens, gather_lens, window_size, compress_ratio, topk, workspace_width,
 * compressed_base) as [BE] _prefill_workspace calls it.
 *
 *   Request r's workspace rows start at r * workspace_width: its compressed
 *   entries 0 .. seq_lens[r]/compress_ratio - 1 at rows 0.., and its gathered
 *   positions g0 = seq_lens[r] - gather_lens[r] .. seq_lens[r] - 1 at rows
 *   compressed_base...  For token t at pos (as combine_topk_swa_indices):
 *   columns [0, W): position max(pos - W + 1, 0) + c -> row
 *     r*ww + compressed_base + (p - g0) when g0 <= p <= pos, else -1;
 *   columns [W, W + topk): local index l -> r*ww + l when
 *     0 <= l < seq_lens[r] / compress_ratio, else -1;
 *   remaining columns up to W + roundup(topk, 4): -1;  lens = entries >= 0.
 *   The column layout is that of combine_topk_swa_indices (the pages do not
 *   print this kernel).  Padding tokens: all -1, lens 0.
 */
psk_status combine_topk_swa_workspace_indices(
    const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* gather_lens, const int32_t* token_to_req, int32_t num_reqs,
    int64_t num_tokens, int32_t window, int32_t compress_ratio,
    const int32_t* topk_local, int64_t topk_stride, int32_t topk,
    int64_t workspace_width, int64_t compressed_base,
    const uint8_t* is_valid_token, int32_t* indices, int64_t out_stride,
    int32_t* lens, psk_stream_t stream);

/*
 * indexer_mxfp4_paged_gather -- raw (packed) MXFP4 rows over request ranges.
 * [MDL] _deepseek_v4_gather_paged_indexer_mxfp4_cache (for the indexer's
 * score GEMM, which reads the packed E2M1 values and E8M0 scales).
 *
 *   values_out   uint8 [total_rows, head_dim/2]; scales_out uint8
 *                [total_rows, head_dim/32] (4-byte aligned rows).
 *   cu_seq_lens  int32 [num_reqs + 1], non-decreasing, cu[0] = 0 and
 *                cu[num_reqs] = total_rows.
 *   Row cu[r] + i holds the record bytes of local position i of request r
 *   through block_table[r] (no base offset), unchanged; a position without a
 *   page gives zero bytes.
 */
psk_status indexer_mxfp4_paged_gather(
    uint8_t* values_out, uint8_t* scales_out, const uint8_t* cache,
    int64_t num_pages, int64_t page_stride, int32_t block_size, int32_t head_dim,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* cu_seq_lens, int32_t num_reqs, int64_t total_rows,
    psk_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Dense builders (TokenSpeed backends/deepseek_v4.py: decode SWA precompute, */
/* HCA dense compressed indices, SWA-only workspace combine)                 */
/* ------------------------------------------------------------------------ */

/*
 * decode_swa_indices_and_lens -- window-only slot indices of decode tokens.
 * TokenSpeed deepseek_v4_decode_swa_indices_and_lens as [BE]
 * _update_decode_swa_metadata calls it (query_start_loc, seq_lens,
 * token_to_req_indices, block_table, block_table_base_offsets, window_size,
 * block_size, is_valid_token).  The kernel is not printed: read as the window
 * columns of combine_topk_swa_indices with no top-k and no replay_start.
 *
 *   out_indices  int32 [num_tokens, window], row stride out_stride (>= window):
 *                column c holds the slot of position lo + c, lo =
 *                max(pos - window + 1, 0), through block_table[r] (logical
 *                page position/block_size - base_offsets[r]), or -1 past pos
 *                or where the page is missing / the slot exceeds INT32_MAX.
 *   out_lens     int32 [num_tokens]: entries >= 0.  Padding tokens
 *                (is_valid_token 0 or a request index outside [0, num_reqs)):
 *                all -1, lens 0.
 *   pos = seq_lens[r] - query_len[r] + (t - query_start_loc[r]).
 */
psk_status decode_swa_indices_and_lens(
    const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* token_to_req, int32_t num_reqs, int64_t num_tokens,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* base_offsets, int32_t block_size, int32_t window,
    const uint8_t* is_valid_token, int32_t* out_indices, int64_t out_stride,
    int32_t* out_lens, psk_stream_t stream);

/*
 * compute_dense_compressed_indices_and_lens -- every visible compressed entry
 * of a decode token (the HCA layers).  [BE]
 * _decode_compressed_attention_indices_and_lens for a compress ratio other
 * than 4 (printed in full).
 *
 *   positions    int64 [num_tokens] token positions (8-byte aligned).
 *   n(t)         = clamp(floor((positions[t] + 1) / compress_ratio), 0, width).
 *   out_indices  int32 [num_tokens, width], row stride out_stride (>= width):
 *                column j holds, for j < n(t), the slot of compressed entry j
 *                through block_table[r] (logical page j/block_size -
 *                base_offsets[r]) or -1 where that page is missing; -1 for
 *                j >= n(t).
 *   out_lens     int32 [num_tokens]: n(t) -- the count of visible entries,
 *                including those whose page is missing, as the pages print
 *                it -- and 0 for a padding token (is_valid_token 0, or a
 *                request index outside [0, num_reqs), whose row is all -1).
 *   width        the caller's dense width (the pages round
 *                ceil(context_len / ratio) up to an alignment).
 */
psk_status compute_dense_compressed_indices_and_lens(
    const int64_t* positions, int64_t num_tokens, const int32_t* token_to_req,
    int32_t num_reqs, const int32_t* block_table, int64_t bt_stride,
    int32_t bt_width, const int32_t* base_offsets, int32_t block_size,
    int32_t compress_ratio, int32_t width, const uint8_t* is_valid_token,
    int32_t* out_indices, int64_t out_stride, int32_t* out_lens,
    psk_stream_t stream);

/*
 * build_dense_prefill_local_compressed_indices -- request-local dense
 * compressed indices of prefill tokens (the HCA prefill workspace's top-k
 * input).  TokenSpeed deepseek_v4_build_dense_prefill_local_compressed_indices
 * (positions, compress_ratio, width, out) as [BE]
 * _dense_prefill_local_compressed_indices calls it; the kernel is not printed:
 * read as out[t][j] = j for j < clamp(floor((positions[t] + 1) / ratio), 0,
 * width), else -1.  out: int32 [num_tokens, width], row stride out_stride.
 */
psk_status build_dense_prefill_local_compressed_indices(
    const int64_t* positions, int64_t num_tokens, int32_t compress_ratio,
    int32_t width, int32_t* out, int64_t out_stride, psk_stream_t stream);

/*
 * combine_dense_swa_indices -- workspace-relative window indices of layers
 * without a compressed cache (compress_ratio <= 1).  TokenSpeed
 * deepseek_v4_combine_dense_swa_indices as [BE] _prefill_workspace calls it
 * (its compressed lengths are then all zero); the kernel is not printed: read
 * as the window columns of combine_topk_swa_workspace_indices with the token's
 * position given.
 *
 *   indices  int32 [num_tokens, window], row stride out_stride (>= window):
 *            column c holds position p = max(positions[t] - window + 1, 0) + c
 *            as workspace row r*workspace_width + compressed_base + (p - g0)
 *            when g0 <= p <= positions[t], g0 = seq_lens[r] - gather_lens[r];
 *            else -1 (also for rows beyond INT32_MAX).
 *   lens     int32 [num_tokens]: entries >= 0.  A request index outside
 *            [0, num_reqs) gives an all -1 row with lens 0.
 */
psk_status combine_dense_swa_indices(
    const int64_t* positions, const int32_t* token_to_req,
    const int32_t* seq_lens, const int32_t* gather_lens, int32_t num_reqs,
    int64_t num_tokens, int32_t window, int64_t workspace_width,
    int64_t compressed_base, int32_t* indices, int64_t out_stride,
    int32_t* lens, psk_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Indexer-key variants: the FP8 indexer record and the fused k_norm ->      */
/* RoPE -> quant -> store of indexer keys                                    */
/* ------------------------------------------------------------------------ */

/*
 * write_indexer_fp8_cache -- FP8 indexer keys in the "[values | fp32 scale]"
 * page layout.  TokenSpeed write_deepseek_v4_indexer_fp8_cache and its
 * capturable form; the rule of _fp8_e4m3_pow2_bytes.
 *
 *   index_k   bf16 [num_tokens, head_dim], row stride k_row_stride (elements,
 *             multiple of 8; 16-byte aligned).
 *   Per token: scale = 2^ceil(log2(max(amax / 448, 1e-10))) (the exact ceiling
 *   of the binary32 quotient), code = e4m3(clamp(x / scale, +-448)).
 *   Page: [block_size x head_dim e4m3 bytes][block_size x 4-byte binary32
 *   scales]; page_stride >= block_size * (head_dim + 4), a multiple of 16.
 *   Slots < 0 are skipped; slots >= num_pages * block_size are skipped and
 *   counted in *err_count (optional).  head_dim in {32, 64, ..., 1024}.
 */
psk_status write_indexer_fp8_cache(
    const void* index_k, int64_t k_row_stride, const int64_t* slot_mapping,
    int64_t num_tokens, uint8_t* cache, int64_t num_pages, int64_t page_stride,
    int32_t block_size, int32_t head_dim, int32_t* err_count, psk_stream_t stream);

/*
 * indexer_k_norm_rope_store -- k_norm -> RoPE -> quant -> paged store of
 * 128-dim indexer keys.  [VLLM] indexer_k_norm_rope_store(k_pre, positions,
 * cos_sin_cache, rms_norm_weight, rms_norm_eps, k_cache, kv_slot_mapping,
 * compress_ratio, use_fp4_cache); its kernel is not printed, so each stage
 * follows the pages' torch form of it.
 *
 *   k_pre            bf16 [num_tokens, 128], row stride k_row_stride (elements,
 *                    multiple of 8; 16-byte aligned).
 *   positions        int64 [num_tokens].
 *   cos_sin_cache    binary32 [max_pos, cs_stride]: 32 cos then 32 sin (GPT-J).
 *   rms_norm_weight  binary32 [128], 16-byte aligned.
 *   Token t writes a key at kv_slot_mapping[t] when that slot is >= 0 and
 *   (positions[t] + 1) % compress_ratio == 0 (it closes its group; other rows
 *   are not read).  Key: x = k_pre[t] in binary32; variance = pairwise sum of
 *   x_d^2 (recursive halving in index order) / 128; r = 1 / sqrt(variance +
 *   rms_norm_eps) as IEEE binary32 square root then division; y = (x * r) * w;
 *   then GPT-J RoPE on dims 64..127 (pair i: y[64+2i], y[65+2i] rotated by
 *   cos_sin_cache[p][i], [p][32+i], p = floor(pos / ratio) * ratio), every
 *   product and sum rounded to binary32 without contraction; then the MXFP4
 *   record (record = PSK_REC_MXFP4, 68-byte keys) or the FP8 indexer record
 *   (PSK_REC_FP8_INDEXER, 132-byte keys), as the two writers above quantize.
 *   Slots >= capacity and RoPE rows p outside [0, max_pos) are skipped and
 *   counted in *err_count (optional).
 */
psk_status indexer_k_norm_rope_store(
    const void* k_pre, int64_t k_row_stride, const int64_t* positions,
    const float* cos_sin_cache, int64_t cs_stride, int64_t max_pos,
    const float* rms_norm_weight, float rms_norm_eps,
    const int64_t* kv_slot_mapping, int64_t num_tokens, int32_t compress_ratio,
    psk_record record, uint8_t* k_cache, int64_t num_pages, int64_t page_stride,
    int32_t block_size, int32_t* err_count, psk_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Compressed-KV producer (TokenSpeed deepseek_v4_ops.py)                     */
/* ------------------------------------------------------------------------ */

/*
 * save_compressor_state -- the compressor's residual state of each token.
 * TokenSpeed save_deepseek_v4_compressor_state: "[kv_state, score_state], each
 * with width coff * head_dim; score state includes the APE row selected by
 * position % compress_ratio".  The kernel is not printed: read as
 * state[slot] = [kv[t], score[t] + ape[pos % ratio]] (binary32 adds).
 *
 *   kv, score    binary32 [num_tokens, in_stride] (16-byte aligned, in_stride a
 *                multiple of 4 >= state_width).
 *   ape          binary32 [compress_ratio, state_width].
 *   state_cache  binary32 [num_pages, block_size, 2 * state_width] (16-byte
 *                aligned); row = slot.
 *   Slots < 0 are skipped; slots >= num_pages * block_size are skipped and
 *   counted in *err_count (optional).
 */
psk_status save_compressor_state(
    const float* kv, const float* score, int64_t in_stride, const float* ape,
    int32_t state_width, const int64_t* slot_mapping, const int64_t* positions,
    int64_t num_tokens, int32_t compress_ratio, float* state_cache, int64_t num_pages,
    int32_t block_size, int32_t* err_count, psk_stream_t stream);

/*
 * compress_kv_cache_insert -- the compressed KV row of every token that closes
 * a compress group, window-pooled from the compressor state, normalised,
 * rotated and inserted as an fp8_ds_mla record (512 dims = 448 + 64 RoPE).
 * TokenSpeed deepseek_v4_csa_compress_kv_cache_insert (compress_ratio 4,
 * overlap 1) and deepseek_v4_hca_compress_kv_cache_insert (128, overlap 0),
 * whose torch form is _compress_v4_state_windows_capturable followed by
 * _write_fp8_ds_mla_cache_rows_capturable.
 *
 *   Token t writes when state_slot_mapping[t] and kv_slot_mapping[t] are >= 0
 *   and (pos + 1) % ratio == 0.  Its window is the W = (overlap ? 2 : 1) *
 *   ratio positions pos - W + 1 + j (W <= 256); position p is present when
 *   p >= 0 and block_table[r][p / state_block_size - base_offsets[r]] (index in
 *   [0, bt_width)) is >= 0; its state row is entry * state_block_size + p %
 *   state_block_size.  Column d of window row j: kv = row[off + d], score =
 *   row[state_width + off + d], off = 512 for j >= ratio under overlap (the
 *   newer positions take the second slice), else 0; absent rows score -1e30
 *   with kv 0.  Per column: m = max_j score; e_j = exp(score_j - m); sum =
 *   e_0 + e_1 + ...; c_d = kv_0 (e_0 / sum) + kv_1 (e_1 / sum) + ... (window
 *   order; binary32, no contraction; exp by Cody-Waite reduction and the Taylor
 *   series to r^7/7!, the oracle's sequence).  Then RMSNorm as
 *   indexer_k_norm_rope_store's (pairwise sum of squares / 512, IEEE sqrt then
 *   reciprocal, (c * r) * weight), GPT-J RoPE of dims 448..511 at
 *   floor(pos / ratio) * ratio, and the fp8_ds_mla record of the bf16 row
 *   (quantize_and_insert_k_cache's UE8M0 rule) at kv_slot_mapping[t].
 *   Slots beyond the kv cache, RoPE rows outside [0, max_pos) and request
 *   indices outside [0, num_reqs) are skipped and counted in *err_count.
 */
psk_status compress_kv_cache_insert(
    const float* state_cache, int64_t state_num_pages, int32_t state_block_size,
    int32_t state_width, const int32_t* token_to_req, const int64_t* positions,
    const int64_t* state_slot_mapping, const int32_t* block_table, int64_t bt_stride,
    int32_t bt_width, const int32_t* base_offsets, int32_t num_reqs, int64_t num_tokens,
    int32_t compress_ratio, int32_t overlap, const float* rms_norm_weight,
    float rms_norm_eps, const float* cos_sin_cache, int64_t cs_stride, int64_t max_pos,
    uint8_t* kv_cache, int64_t kv_num_pages, int64_t kv_page_stride,
    int32_t kv_block_size, const int64_t* kv_slot_mapping, int32_t* err_count,
    psk_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Fused gathers: the slots computed in the gather (no index matrix)          */
/* ------------------------------------------------------------------------ */

/*
 * dequantize_and_gather_k_cache_topk -- the top-k columns of a token gathered
 * straight from its local top-k indices.  Output identical to
 * compute_global_topk_indices_and_lens (table, base offsets, padding tokens)
 * followed by dequantize_and_gather_k_cache over that matrix, in one launch
 * with no index matrix in between (the pages' decode path maps local top-k to
 * global slots, [BE] _decode_compressed_attention_indices_and_lens, then the
 * attention reads those rows; here the rows are dequantised directly).
 *
 *   out           bf16 rows (t, j) at out + t*out_stride_t + j*out_stride_j,
 *                 j < topk (elements, multiples of 8).
 *   topk_local    int32 [num_tokens, topk_stride].
 *   record        any of the three; fp8_ds_mla with UE8M0 scales.
 *   Arguments as in compute_global_topk_indices_and_lens and
 *   dequantize_and_gather_k_cache.
 */
psk_status dequantize_and_gather_k_cache_topk(
    void* out, int64_t out_stride_t, int64_t out_stride_j, const uint8_t* cache,
    int64_t num_pages, int64_t page_stride, int32_t block_size, psk_record record,
    int32_t head_dim, int32_t rope_dim, const int32_t* topk_local, int64_t topk_stride,
    int64_t num_tokens, int32_t topk, const int32_t* token_to_req,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width, int32_t num_reqs,
    const int32_t* base_offsets, const uint8_t* is_valid_token, psk_stream_t stream);

/*
 * dequantize_and_gather_k_cache_window -- the window columns of a token
 * gathered straight from its position.  Output identical to the window
 * columns [0, window) of combine_topk_swa_indices (position from the
 * metadata, window [max(replay_start, pos - window + 1, 0), pos] left-aligned,
 * the SWA table and base offsets, padding tokens) followed by
 * dequantize_and_gather_k_cache over them, in one launch.  fp8_ds_mla records
 * with UE8M0 scales; out rows (t, c), c < window, as above.
 */
psk_status dequantize_and_gather_k_cache_window(
    void* out, int64_t out_stride_t, int64_t out_stride_j, const uint8_t* cache,
    int64_t num_pages, int64_t page_stride, int32_t block_size, int32_t head_dim,
    int32_t rope_dim, const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* token_to_req, const int32_t* replay_start, int32_t num_reqs,
    int64_t num_tokens, const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* base_offsets, int32_t window, const uint8_t* is_valid_token,
    psk_stream_t stream);

/*
 * dequantize_and_gather_k_cache_pair -- one index matrix read against two
 * fp8_ds_mla caches of the same record format: columns j < split take their
 * slots in cache_a, columns j >= split in cache_b.  This is how the decode
 * attention reads the combined matrix of combine_topk_swa_indices against
 * the SWA cache (window columns) and the compressed cache (top-k columns),
 * [BE] forward_deepseek_v4_decode (k_cache with extra_k_cache); the output
 * equals dequantize_and_gather_k_cache over columns [0, split) of cache_a and
 * over columns [split, cols) of cache_b, in one launch.  UE8M0 scales; each
 * cache has its own pages, page stride and block size; slots outside a cache
 * give zero rows as in dequantize_and_gather_k_cache.
 *
 *   out      bf16 rows (t, j) at out + t*out_stride_t + j*out_stride_j,
 *            j < cols (elements, multiples of 8; 16-byte aligned).
 *   indices  int32 [rows, idx_stride], idx_stride >= cols.
 *   split    0 <= split <= cols.
 *   Errors: PSK_ERR_INVALID_ARGUMENT as dequantize_and_gather_k_cache, for
 *   either cache; PSK_ERR_CUDA if the launch fails.
 */
psk_status dequantize_and_gather_k_cache_pair(
    void* out, int64_t out_stride_t, int64_t out_stride_j, const uint8_t* cache_a,
    int64_t num_pages_a, int64_t page_stride_a, int32_t block_size_a, const uint8_t* cache_b,
    int64_t num_pages_b, int64_t page_stride_b, int32_t block_size_b, int32_t head_dim,
    int32_t rope_dim, const int32_t* indices, int64_t idx_stride, int64_t rows, int32_t cols,
    int32_t split, psk_stream_t stream);

/*
 * dequantize_and_gather_k_cache_dense -- every visible compressed entry of a
 * token gathered straight from its position (the HCA decode read of a heavily
 * compressed layer, [BE] _decode_compressed_attention_indices_and_lens with
 * all (pos + 1) // ratio entries).  Output identical to
 * compute_dense_compressed_indices_and_lens (same arguments) followed by
 * dequantize_and_gather_k_cache over that matrix, in one launch: out row
 * (t, c), c < width, is compressed entry c when c < clamp((positions[t] + 1)
 * // compress_ratio, 0, width) and the token is valid, else a zero row.
 * fp8_ds_mla records with UE8M0 scales; out as in
 * dequantize_and_gather_k_cache_topk.  Errors: PSK_ERR_INVALID_ARGUMENT as the
 * two calls it stands for; PSK_ERR_CUDA if the launch fails.
 */
psk_status dequantize_and_gather_k_cache_dense(
    void* out, int64_t out_stride_t, int64_t out_stride_j, const uint8_t* cache,
    int64_t num_pages, int64_t page_stride, int32_t block_size, int32_t head_dim,
    int32_t rope_dim, const int64_t* positions, int64_t num_tokens, const int32_t* token_to_req,
    int32_t num_reqs, const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* base_offsets, int32_t compress_ratio, int32_t width,
    const uint8_t* is_valid_token, psk_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PSK_H */
