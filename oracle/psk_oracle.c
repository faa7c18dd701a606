/*
 * psk_oracle.c -- CPU oracle for the paged sparse K-cache pipeline.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this file's library.  The product
 * library never includes, links or calls it, and this file includes nothing
 * from the product library: the two implementations share no code.
 *
 * Plain, slow, single-threaded C.  Each step follows the statement it cites,
 * in the order the statement gives, with no blocking or fusion.  Floating
 * point is IEEE binary32 with round-to-nearest-even, as the pages' torch
 * restatements compute it; build without fast-math and without FMA
 * contraction so the host rounds every operation once.
 *
 * Sources (page title, then the section/function on it):
 *   [OPS]  TokenSpeed runtime/layers/attention/deepseek_v4_ops.py
 *   [BE]   TokenSpeed runtime/layers/attention/backends/deepseek_v4.py
 *   [MDL]  TokenSpeed runtime/models/deepseek_v4.py
 *   [VLLM] vLLM API docs, vllm.models.deepseek_v41.common.ops
 *   [OFP8] OCP 8-bit Floating Point Specification (OFP8), E4M3 encoding
 *   [MX]   OCP Microscaling Formats (MX) v1.0, E2M1 element and E8M0 scale
 *
 * Parity pins live in tests/test_oracle_*.py.  The fp32-scale FP8 record
 * (is_ue8m0 = 0) is printed on no page; its rule (scale = max(amax, 1e-12) /
 * 448 and the codes of x / scale, both IEEE binary32 divisions) is pinned by a
 * hand-worked golden record (insert and gather) and against torch's e4m3
 * encode and decode.
 */
#include "psk_oracle.h"

#include <math.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                             */
/* ------------------------------------------------------------------------ */

/* Round a non-negative double to the nearest integer, ties to even. */
static double round_half_even(double q) {
    double f = floor(q);
    double frac = q - f;
    if (frac > 0.5) return f + 1.0;
    if (frac < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/*
 * [OFP8] E4M3 ("FN" variant): sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; no infinities; S.1111.111 is NaN; the largest finite magnitude is
 * 1.75 * 2^8 = 448.  Exponent field 0 holds subnormals m * 2^-9.
 * Rounding is to nearest, ties to even; magnitudes beyond 448 saturate to 448
 * (the "satfinite" conversion).  The sign of zero is kept.
 */
uint8_t oracle_e4m3_encode(float v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range, spacing 2^-9; a count of 8 is the smallest normal
         * (exponent field 1, mantissa 0), which is also code 8. */
        double m = round_half_even(a * 512.0);
        return sign | (uint8_t)m;
    }
    int ex;
    (void)frexp(a, &ex);
    int e = ex - 1; /* 2^e <= a < 2^(e+1), e in [-6, 8] */
    double m = round_half_even(ldexp(a, 3 - e)); /* significand * 8, in [8, 16] */
    if (m == 16.0) {
        e += 1;
        m = 8.0;
    }
    int code = ((e + 7) << 3) | ((int)m - 8);
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

float oracle_e4m3_decode(uint8_t code) {
    int s = code >> 7, e = (code >> 3) & 0xF, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (float)(s ? -v : v);
}

/*
 * [MX] E2M1: sign bit, 2 exponent bits (bias 1), 1 mantissa bit.  Magnitudes
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}; no infinities or NaN.  Round to nearest, ties
 * to the even code; saturate to 6; keep the sign of zero.
 */
uint8_t oracle_e2m1_encode(float v) {
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs((double)v);
    if (isnan(v)) return 0x7;
    if (a >= 6.0) return sign | 0x7;
    if (a < 1.0) {
        /* exponent field 0: subnormal 0.5 * m; a count of 2 is 1.0 = code 2 */
        double m = round_half_even(a * 2.0);
        return sign | (uint8_t)m;
    }
    int ex;
    (void)frexp(a, &ex);
    int e = ex - 1; /* e in [0, 2] */
    double m = round_half_even(ldexp(a, 1 - e)); /* significand * 2, in [2, 4] */
    if (m == 4.0) {
        e += 1;
        m = 2.0;
    }
    if (e > 2) return sign | 0x7;
    return sign | (uint8_t)(((e + 1) << 1) | ((int)m - 2));
}

float oracle_e2m1_decode(uint8_t nibble) {
    int s = (nibble >> 3) & 1, e = (nibble >> 1) & 3, f = nibble & 1;
    double v = (e == 0) ? 0.5 * f : ldexp((double)(2 + f), e - 2);
    return (float)(s ? -v : v);
}

/*
 * Smallest integer e with 2^e >= q, for finite q > 0 (exact; no log2 call).
 * frexp gives q = f * 2^ex with f in [0.5, 1): q is a power of two exactly
 * when f == 0.5, and then e = ex - 1; otherwise e = ex.
 */
int32_t oracle_ceil_log2(float q) {
    if (isinf(q)) return 128;
    int ex;
    double f = frexp((double)q, &ex);
    return (f == 0.5) ? ex - 1 : ex;
}

/* bf16 is the upper half of binary32.  Rounding to bf16 drops 16 low bits,
 * to nearest with ties to even; NaN maps to the canonical quiet NaN. */
uint16_t oracle_bf16_from_f32(float f) {
    if (isnan(f)) return 0x7FFF;
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

float oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

void oracle_e4m3_encode_array(const float* v, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

void oracle_e2m1_encode_array(const float* v, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_encode(v[i]);
}

void oracle_ceil_log2_array(const float* q, int32_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_ceil_log2(q[i]);
}

/* 2^k as binary32: exact for k in [-149, 127], +inf above, 0 below. */
static float pow2f(int k) {
    if (k > 127) return INFINITY;
    if (k < -149) return 0.0f;
    return ldexpf(1.0f, k);
}

/* ------------------------------------------------------------------------ */
/* Record geometry                                                            */
/* ------------------------------------------------------------------------ */

/*
 * fp8_ds_mla record ([OPS] dequantize_deepseek_v4_fp8_ds_mla_cache and
 * _fp8_ds_mla_cache_rows; [VLLM] quantize_and_insert_k_cache): per token the
 * nope dims as one e4m3 byte each, then the rope dims as bf16 (2 bytes each);
 * after block_size such data records, block_size scale records.  Quant blocks
 * are 64 wide; a token carries head_dim/64 scale slots (448 + 64 -> 7 used +
 * 1 zero pad = 8, as the insert docs fix for head_dim 512).
 */
int64_t oracle_fp8_token_stride(int32_t head_dim, int32_t rope_dim) {
    return (int64_t)(head_dim - rope_dim) + 2 * (int64_t)rope_dim;
}

int64_t oracle_fp8_scale_bytes(int32_t head_dim, int32_t is_ue8m0) {
    /* one UE8M0 byte per 64-block, or one little-endian binary32 per block */
    return (int64_t)(head_dim / 64) * (is_ue8m0 ? 1 : 4);
}

/* ------------------------------------------------------------------------ */
/* Step 1a: FP8 quantize-and-insert                                           */
/* ------------------------------------------------------------------------ */

/*
 * [VLLM] quantize_and_insert_k_cache; the math is [OPS] _fp8_ds_mla_cache_rows
 * and its writer _write_fp8_ds_mla_cache_rows_capturable.
 *
 * For every token i with slot s = slot_mapping[i]:
 *   s < 0 is skipped (padding); s >= num_pages * block_size is skipped and
 *   counted (fail closed, [MDL] _deepseek_v4_swa_slot_mapping).
 *   page = s / block_size, off = s % block_size.
 *   For each 64-wide block of the nope dims:
 *     is_ue8m0 = 1 (the pages' rule):
 *       amax = max |x|, floored at 1e-4;
 *       e = ceil(log2(amax / 448)) taken exactly on the binary32 quotient;
 *       scale byte = clamp(e + 127, 0, 255);
 *       code = e4m3(clamp(x * 2^-e, -448, 448)).
 *     is_ue8m0 = 0 (fp32 scales, not on the pages):
 *       scale = max(amax, 1e-12) / 448 (binary32, stored little-endian);
 *       code = e4m3(clamp(x / scale, -448, 448)).
 *   The rope dims are copied as bf16 bit patterns; unused scale slots are 0.
 * Returns the number of out-of-range slots.
 */
int64_t oracle_quantize_and_insert_k_cache(
    const uint16_t* k, int64_t k_row_stride, const int64_t* slot_mapping,
    int64_t num_tokens, uint8_t* cache, int64_t num_pages,
    int64_t page_stride, int32_t block_size, int32_t head_dim,
    int32_t rope_dim, int32_t is_ue8m0) {
    const int32_t nope = head_dim - rope_dim;
    const int64_t ts = oracle_fp8_token_stride(head_dim, rope_dim);
    const int64_t sdim = oracle_fp8_scale_bytes(head_dim, is_ue8m0);
    const int32_t nblk = nope / 64;
    const int64_t capacity = num_pages * (int64_t)block_size;
    int64_t errors = 0;

    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t s = slot_mapping[i];
        if (s < 0) continue;
        if (s >= capacity) {
            ++errors;
            continue;
        }
        const int64_t page = s / block_size, off = s % block_size;
        uint8_t* data = cache + page * page_stride + off * ts;
        uint8_t* scl = cache + page * page_stride + (int64_t)block_size * ts + off * sdim;
        const uint16_t* row = k + i * k_row_stride;

        memset(scl, 0, (size_t)sdim);
        for (int32_t b = 0; b < nblk; ++b) {
            float x[64];
            float amax = 0.0f;
            for (int j = 0; j < 64; ++j) {
                x[j] = oracle_bf16_to_f32(row[b * 64 + j]);
                float a = fabsf(x[j]);
                if (a > amax) amax = a;
            }
            if (is_ue8m0) {
                float a = (amax < 1.0e-4f) ? 1.0e-4f : amax;
                float q = a / 448.0f;
                int32_t e = oracle_ceil_log2(q);
                int32_t byte = e + 127;
                if (byte < 0) byte = 0;
                if (byte > 255) byte = 255;
                scl[b] = (uint8_t)byte;
                float p = pow2f(-e);
                for (int j = 0; j < 64; ++j) {
                    float v = x[j] * p;
                    if (v > 448.0f) v = 448.0f;
                    if (v < -448.0f) v = -448.0f;
                    data[b * 64 + j] = oracle_e4m3_encode(v);
                }
            } else {
                float a = (amax < 1.0e-12f) ? 1.0e-12f : amax;
                float scale = a / 448.0f;
                memcpy(scl + 4 * b, &scale, 4);
                for (int j = 0; j < 64; ++j) {
                    float v = x[j] / scale;
                    if (v > 448.0f) v = 448.0f;
                    if (v < -448.0f) v = -448.0f;
                    data[b * 64 + j] = oracle_e4m3_encode(v);
                }
            }
        }
        /* rope tail: bf16 bit patterns, verbatim (already rotated by the caller) */
        memcpy(data + nope, row + nope, (size_t)rope_dim * 2);
    }
    return errors;
}

/* ------------------------------------------------------------------------ */
/* Step 1b: MXFP4 indexer-key insert                                          */
/* ------------------------------------------------------------------------ */

/*
 * [OPS] write_deepseek_v4_indexer_mxfp4_cache (page layout) and
 * read_deepseek_v4_indexer_mxfp4_cache (the inverse that fixes nibble order
 * and scale meaning).  The writer's scale rule is not printed; the reading
 * taken is E8M0 = ceil-pow2(amax / 6), with amax floored at 1e-4 as the FP8
 * writer floors it.
 *
 * Per token and 32-wide block: e = ceil(log2(max(amax, 1e-4) / 6)),
 * scale byte = clamp(e + 127, 0, 254), code = e2m1(x * 2^-e) (saturating).
 * Byte j of the values holds element 2j in its low nibble and 2j+1 in its
 * high nibble.  Page: [block_size x head_dim/2 value bytes]
 * [block_size x head_dim/32 scale bytes].
 */
int64_t oracle_write_indexer_mxfp4_cache(
    const uint16_t* k, int64_t k_row_stride, const int64_t* slot_mapping,
    int64_t num_tokens, uint8_t* cache, int64_t num_pages,
    int64_t page_stride, int32_t block_size, int32_t head_dim) {
    const int64_t vbytes = head_dim / 2, sbytes = head_dim / 32;
    const int64_t capacity = num_pages * (int64_t)block_size;
    int64_t errors = 0;

    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t s = slot_mapping[i];
        if (s < 0) continue;
        if (s >= capacity) {
            ++errors;
            continue;
        }
        const int64_t page = s / block_size, off = s % block_size;
        uint8_t* vals = cache + page * page_stride + off * vbytes;
        uint8_t* scl = cache + page * page_stride + (int64_t)block_size * vbytes + off * sbytes;
        const uint16_t* row = k + i * k_row_stride;

        for (int32_t b = 0; b < head_dim / 32; ++b) {
            float x[32];
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j) {
                x[j] = oracle_bf16_to_f32(row[b * 32 + j]);
                float a = fabsf(x[j]);
                if (a > amax) amax = a;
            }
            float a = (amax < 1.0e-4f) ? 1.0e-4f : amax;
            float q = a / 6.0f;
            int32_t e = oracle_ceil_log2(q);
            int32_t byte = e + 127;
            if (byte < 0) byte = 0;
            if (byte > 254) byte = 254;
            scl[b] = (uint8_t)byte;
            float p = pow2f(-e);
            for (int j = 0; j < 32; j += 2) {
                uint8_t lo = oracle_e2m1_encode(x[j] * p);
                uint8_t hi = oracle_e2m1_encode(x[j + 1] * p);
                vals[(b * 32 + j) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    return errors;
}

/* ------------------------------------------------------------------------ */
/* Step 2: index builders                                                     */
/* ------------------------------------------------------------------------ */

/*
 * Slot of logical position `pos` through one request's block-table row
 * ([MDL] indexer prefill gather plan: page_ids * block_size + offset;
 * [BE] dense compressed indices with safe_page_ids; [OPS]
 * _compress_v4_state_windows_capturable for the base_logical_page offset and
 * the validity rules):
 *   logical page = pos / block_size - base;  outside [0, width) -> -1;
 *   page id = row[logical page];  page id < 0 -> -1;
 *   slot = page id * block_size + pos % block_size  (-1 if beyond int32).
 */
static int32_t slot_of(const int32_t* row, int32_t width, int64_t base,
                       int32_t block_size, int64_t pos) {
    if (pos < 0) return -1;
    int64_t lp = pos / block_size - base;
    if (lp < 0 || lp >= width) return -1;
    int32_t page = row[lp];
    if (page < 0) return -1;
    int64_t s = (int64_t)page * block_size + pos % block_size;
    if (s > INT32_MAX) return -1;
    return (int32_t)s;
}

/*
 * [VLLM] compute_global_topk_indices_and_lens: per token, map every local
 * top-k index through the token's request block table; -1 stays -1; count the
 * valid entries into lens; an invalid (padding) token gets lens 0 and, in the
 * reading taken here, all of its entries written as -1.  A token whose request
 * index is outside [0, num_reqs) is treated as invalid.  Entries are not
 * compacted.
 */
void oracle_compute_global_topk_indices_and_lens(
    const int32_t* topk_local, int64_t topk_stride, int64_t num_tokens,
    int32_t topk, const int32_t* token_to_req, const int32_t* block_table,
    int64_t bt_stride, int32_t bt_width, int32_t num_reqs, int32_t block_size,
    const int32_t* base_offsets, const uint8_t* is_valid_token,
    int32_t* out_indices, int64_t out_stride, int32_t* out_lens) {
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int32_t r = token_to_req[t];
        const int ok = (is_valid_token ? is_valid_token[t] != 0 : 1) &&
                       r >= 0 && r < num_reqs;
        int32_t count = 0;
        for (int32_t j = 0; j < topk; ++j) {
            int32_t v = -1;
            if (ok) {
                int32_t l = topk_local[t * topk_stride + j];
                if (l >= 0) {
                    int64_t base = base_offsets ? base_offsets[r] : 0;
                    v = slot_of(block_table + (int64_t)r * bt_stride, bt_width,
                                base, block_size, l);
                }
            }
            out_indices[t * out_stride + j] = v;
            if (v >= 0) ++count;
        }
        out_lens[t] = count;
    }
}

/*
 * [VLLM] build_flashinfer_mixed_sparse_indices (the single-kernel form of
 * TokenSpeed's combine_topk_swa_indices).  Per token t of request r:
 *   position  pos = seq_lens[r] - query_len[r] + (t - query_start_loc[r])
 *             ([BE] _decode_positions_from_metadata);
 *   window    [lo, pos] with lo = max(replay_start[r], pos - window + 1, 0);
 *   columns [0, window): column c holds the slot of position lo + c through
 *             the SWA table, or -1 once lo + c > pos (left-aligned, oldest
 *             first -- a reading);
 *   columns [window, window + topk): local top-k index j mapped through the
 *             compressed table (the SWA table when none is given);
 *   columns up to window + roundup(topk, 4): -1 (16-byte row alignment);
 *   lens[t] = number of entries >= 0 over all columns (a reading: the docs
 *             call it the active length per token).
 * replay_start applies to every token (null = 0).  compress_ratio is accepted
 * for the signature and does not change the result (a reading).
 */
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
    int32_t* lens) {
    (void)compress_ratio;
    const int32_t padded = (topk + 3) / 4 * 4;
    const int32_t width = window + padded;
    if (comp_block_table == NULL) {
        comp_block_table = swa_block_table;
        comp_bt_stride = swa_bt_stride;
        comp_bt_width = swa_bt_width;
    }
    for (int64_t t = 0; t < num_tokens; ++t) {
        int32_t* row = sparse_indices + t * out_stride;
        const int32_t r = token_to_req[t];
        const int ok = (is_valid_token ? is_valid_token[t] != 0 : 1) &&
                       r >= 0 && r < num_reqs;
        if (!ok) {
            for (int32_t c = 0; c < width; ++c) row[c] = -1;
            lens[t] = 0;
            continue;
        }
        const int64_t qstart = query_start_loc[r];
        const int64_t qlen = (int64_t)query_start_loc[r + 1] - qstart;
        const int64_t pos = (int64_t)seq_lens[r] - qlen + (t - qstart);
        int64_t lo = pos - window + 1;
        const int64_t rs = replay_start ? replay_start[r] : 0;
        if (rs > lo) lo = rs;
        if (lo < 0) lo = 0;

        int32_t count = 0;
        const int32_t* swa_row = swa_block_table + (int64_t)r * swa_bt_stride;
        const int64_t swa_base = swa_base_offsets ? swa_base_offsets[r] : 0;
        for (int32_t c = 0; c < window; ++c) {
            int64_t p = lo + c;
            int32_t v = (p <= pos) ? slot_of(swa_row, swa_bt_width, swa_base,
                                             swa_block_size, p)
                                   : -1;
            row[c] = v;
            if (v >= 0) ++count;
        }
        const int32_t* comp_row = comp_block_table + (int64_t)r * comp_bt_stride;
        const int64_t comp_base = comp_base_offsets ? comp_base_offsets[r] : 0;
        for (int32_t j = 0; j < topk; ++j) {
            int32_t l = topk_local[t * topk_stride + j];
            int32_t v = (l >= 0) ? slot_of(comp_row, comp_bt_width, comp_base,
                                           comp_block_size, l)
                                 : -1;
            row[window + j] = v;
            if (v >= 0) ++count;
        }
        for (int32_t j = topk; j < padded; ++j) row[window + j] = -1;
        lens[t] = count;
    }
}

/* ------------------------------------------------------------------------ */
/* Step 3: dequantize-and-gather                                              */
/* ------------------------------------------------------------------------ */

/*
 * Index form of the gather: [OPS] dequantize_deepseek_v4_fp8_ds_mla_cache
 * (record 0) and read_deepseek_v4_indexer_mxfp4_cache (record 1), with the
 * rows laid out as out[t][j][d] = out + t*out_stride_t + j*out_stride_j + d.
 *   s = indices[t][j]; s < 0 or s >= capacity -> an all-zero bf16 row.
 *   fp8_ds_mla: nope dim d -> bf16(e4m3(byte d) * 2^(scale[d/64] - 127)) (UE8M0)
 *               or bf16(e4m3(byte d) * scale_f32[d/64]) (fp32 scales);
 *               rope dims -> the stored bf16 bit patterns.
 *   MXFP4:      dim d -> bf16(e2m1(nibble d) * 2^(scale[d/32] - 127)), nibble
 *               d is the low half of byte d/2 for even d, the high half for odd.
 *   FP8 indexer (record 2, [OPS] write_deepseek_v4_indexer_fp8_cache):
 *               dim d -> bf16(e4m3(byte d) * scale_f32).
 * Products are formed in binary32 and rounded once more to bf16.
 */
void oracle_dequantize_and_gather_k_cache(
    uint16_t* out, int64_t out_stride_t, int64_t out_stride_j,
    const uint8_t* cache, int64_t num_pages, int64_t page_stride,
    int32_t block_size, int32_t record, int32_t head_dim, int32_t rope_dim,
    int32_t is_ue8m0, const int32_t* indices, int64_t idx_stride, int64_t rows,
    int32_t cols) {
    const int64_t capacity = num_pages * (int64_t)block_size;
    for (int64_t t = 0; t < rows; ++t) {
        for (int32_t j = 0; j < cols; ++j) {
            const int64_t s = indices[t * idx_stride + j];
            uint16_t* o = out + t * out_stride_t + (int64_t)j * out_stride_j;
            if (s < 0 || s >= capacity) {
                for (int32_t d = 0; d < head_dim; ++d) o[d] = 0;
                continue;
            }
            const int64_t page = s / block_size, off = s % block_size;
            const uint8_t* base = cache + page * page_stride;
            if (record == 0) {
                const int32_t nope = head_dim - rope_dim;
                const int64_t ts = oracle_fp8_token_stride(head_dim, rope_dim);
                const int64_t sdim = oracle_fp8_scale_bytes(head_dim, is_ue8m0);
                const uint8_t* data = base + off * ts;
                const uint8_t* scl = base + (int64_t)block_size * ts + off * sdim;
                for (int32_t d = 0; d < nope; ++d) {
                    float val = oracle_e4m3_decode(data[d]);
                    float f;
                    if (is_ue8m0) {
                        f = val * pow2f((int)scl[d / 64] - 127);
                    } else {
                        float sc;
                        memcpy(&sc, scl + 4 * (d / 64), 4);
                        f = val * sc;
                    }
                    o[d] = oracle_bf16_from_f32(f);
                }
                for (int32_t d = nope; d < head_dim; ++d) {
                    const uint8_t* p = data + nope + 2 * (int64_t)(d - nope);
                    o[d] = (uint16_t)(p[0] | (p[1] << 8));
                }
            } else if (record == 1) {
                const int64_t vbytes = head_dim / 2, sbytes = head_dim / 32;
                const uint8_t* vals = base + off * vbytes;
                const uint8_t* scl = base + (int64_t)block_size * vbytes + off * sbytes;
                for (int32_t d = 0; d < head_dim; ++d) {
                    uint8_t byte = vals[d / 2];
                    uint8_t nib = (d % 2) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
                    float f = oracle_e2m1_decode(nib) * pow2f((int)scl[d / 32] - 127);
                    o[d] = oracle_bf16_from_f32(f);
                }
            } else {
                /* FP8 indexer record: head_dim e4m3 bytes, one binary32 scale */
                const uint8_t* vals = base + off * head_dim;
                float sc;
                memcpy(&sc, base + (int64_t)block_size * head_dim + off * 4, 4);
                for (int32_t d = 0; d < head_dim; ++d)
                    o[d] = oracle_bf16_from_f32(oracle_e4m3_decode(vals[d]) * sc);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Prefill workspace path: range gather, workspace indices, raw MXFP4 gather  */
/* ------------------------------------------------------------------------ */

/*
 * Range form of the gather ([VLLM] dequantize_and_gather_k_cache(out, k_cache,
 * seq_lens, gather_lens, block_table, block_size, offset); called twice per
 * layer by [BE] _prefill_workspace, compressed rows at offset 0 and window rows
 * at offset compressed_base).  For request r, with g = gather_lens[r] (or
 * seq_lens[r] when gather_lens is NULL), row i in [0, g) is position
 * p = seq_lens[r] - g + i, mapped through the request's block-table row, and
 * goes to out[r][offset + i] (dequantized as in the index form; a missing page
 * gives a zero row).  Rows outside [offset, offset + g), and rows at or beyond
 * out_rows, are not written.
 */
void oracle_dequantize_and_gather_k_cache_ranges(
    uint16_t* out, int64_t out_stride_r, int64_t out_stride_i, int64_t out_rows,
    const uint8_t* cache, int64_t num_pages, int64_t page_stride,
    int32_t block_size, int32_t record, int32_t head_dim, int32_t rope_dim,
    int32_t is_ue8m0, const int32_t* seq_lens, const int32_t* gather_lens,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* base_offsets, int32_t num_reqs, int64_t offset) {
    for (int32_t r = 0; r < num_reqs; ++r) {
        const int64_t seq = seq_lens[r];
        const int64_t g = gather_lens ? gather_lens[r] : seq;
        const int64_t base = base_offsets ? base_offsets[r] : 0;
        for (int64_t i = 0; i < g; ++i) {
            if (offset + i < 0 || offset + i >= out_rows) continue;
            const int64_t p = seq - g + i;
            const int32_t s = slot_of(block_table + (int64_t)r * bt_stride, bt_width, base,
                                      block_size, p);
            /* one row through the index-form gather of that slot */
            oracle_dequantize_and_gather_k_cache(
                out + r * out_stride_r + (offset + i) * out_stride_i, 0, 0, cache, num_pages,
                page_stride, block_size, record, head_dim, rope_dim, is_ue8m0, &s, 1, 1, 1);
        }
    }
}

/*
 * Workspace-relative form of the fused index build (TokenSpeed's
 * combine_topk_swa_indices as called by [BE] _prefill_workspace with
 * workspace_width and compressed_base).  Request r's workspace rows start at
 * r * workspace_width: its compressed entries 0 .. floor(seq_lens[r] / ratio) - 1
 * at rows 0.., its gathered window positions g0 .. seq_lens[r] - 1 at rows
 * compressed_base.., with g0 = seq_lens[r] - gather_lens[r].  For token t at
 * pos (as in the global-slot builder):
 *   columns [0, W): position lo + c, lo = max(pos - W + 1, 0), maps to row
 *     r*ww + compressed_base + (p - g0) when g0 <= p <= pos, else -1;
 *   columns [W, W + topk): local index l maps to r*ww + l when
 *     0 <= l < floor(seq_lens[r] / ratio), else -1;
 *   padding to W + roundup(topk, 4): -1;  lens = entries >= 0.
 * Same column layout as the global-slot builder (a reading: the kernel body is
 * not printed).  A padding token is all -1 with lens 0.
 */
void oracle_combine_topk_swa_workspace_indices(
    const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* gather_lens, const int32_t* token_to_req, int32_t num_reqs,
    int64_t num_tokens, int32_t window, int32_t compress_ratio,
    const int32_t* topk_local, int64_t topk_stride, int32_t topk,
    int64_t workspace_width, int64_t compressed_base,
    const uint8_t* is_valid_token, int32_t* indices, int64_t out_stride,
    int32_t* lens) {
    const int32_t padded = (topk + 3) / 4 * 4;
    const int32_t width = window + padded;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int32_t* row = indices + t * out_stride;
        const int32_t r = token_to_req[t];
        const int ok = (is_valid_token ? is_valid_token[t] != 0 : 1) &&
                       r >= 0 && r < num_reqs;
        if (!ok) {
            for (int32_t c = 0; c < width; ++c) row[c] = -1;
            lens[t] = 0;
            continue;
        }
        const int64_t qstart = query_start_loc[r];
        const int64_t qlen = (int64_t)query_start_loc[r + 1] - qstart;
        const int64_t seq = seq_lens[r];
        const int64_t pos = seq - qlen + (t - qstart);
        const int64_t g0 = seq - gather_lens[r];
        const int64_t lc = seq / compress_ratio;
        const int64_t rbase = (int64_t)r * workspace_width;
        int64_t lo = pos - window + 1;
        if (lo < 0) lo = 0;
        int32_t count = 0;
        for (int32_t c = 0; c < window; ++c) {
            const int64_t p = lo + c;
            int64_t v = -1;
            if (p <= pos && p >= g0) v = rbase + compressed_base + (p - g0);
            if (v > INT32_MAX) v = -1;
            row[c] = (int32_t)v;
            if (v >= 0) ++count;
        }
        for (int32_t j = 0; j < topk; ++j) {
            const int64_t l = topk_local[t * topk_stride + j];
            int64_t v = (l >= 0 && l < lc) ? rbase + l : -1;
            if (v > INT32_MAX) v = -1;
            row[window + j] = (int32_t)v;
            if (v >= 0) ++count;
        }
        for (int32_t j = topk; j < padded; ++j) row[window + j] = -1;
        lens[t] = count;
    }
}

/*
 * Raw (packed) gather of MXFP4 indexer keys over per-request ranges
 * ([MDL] _deepseek_v4_gather_paged_indexer_mxfp4_cache -> indexer_mxfp4_paged_gather):
 * output row cu_seq_lens[r] + i (i < cu_seq_lens[r+1] - cu_seq_lens[r]) holds the
 * head_dim/2 value bytes and head_dim/32 scale bytes of local position i of
 * request r, copied unchanged; a position without a page gives zero bytes.
 */
void oracle_indexer_mxfp4_paged_gather(
    uint8_t* values_out, uint8_t* scales_out, const uint8_t* cache,
    int64_t num_pages, int64_t page_stride, int32_t block_size,
    int32_t head_dim, const int32_t* block_table, int64_t bt_stride,
    int32_t bt_width, const int32_t* cu_seq_lens, int32_t num_reqs) {
    const int64_t vb = head_dim / 2, sb = head_dim / 32;
    const int64_t capacity = num_pages * (int64_t)block_size;
    for (int32_t r = 0; r < num_reqs; ++r) {
        for (int64_t row = cu_seq_lens[r]; row < cu_seq_lens[r + 1]; ++row) {
            const int64_t i = row - cu_seq_lens[r];
            const int32_t s = slot_of(block_table + (int64_t)r * bt_stride, bt_width, 0,
                                      block_size, i);
            uint8_t* vo = values_out + row * vb;
            uint8_t* so = scales_out + row * sb;
            if (s < 0 || s >= capacity) {
                memset(vo, 0, (size_t)vb);
                memset(so, 0, (size_t)sb);
                continue;
            }
            const int64_t page = s / block_size, off = s % block_size;
            const uint8_t* base = cache + page * page_stride;
            memcpy(vo, base + off * vb, (size_t)vb);
            memcpy(so, base + (int64_t)block_size * vb + off * sb, (size_t)sb);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Dense builders: decode SWA indices, HCA dense compressed indices, dense   */
/* prefill local indices, SWA-only workspace combine                        */
/* ------------------------------------------------------------------------ */

/*
 * [OPS] deepseek_v4_decode_swa_indices_and_lens as [BE]
 * _update_decode_swa_metadata calls it (query_start_loc, seq_lens,
 * token_to_req_indices, block_table, block_table_base_offsets, window_size,
 * block_size, is_valid_token -> indices [T, window_size], lens [T]).  The body
 * is not printed; read as the window part of the fused builder: the token's
 * position from the metadata ([BE] _decode_positions_from_metadata), window
 * [max(pos - window + 1, 0), pos] left-aligned, oldest first; each position's
 * slot through the SWA table (minus the request's base logical page) or -1;
 * lens = entries >= 0; a padding token (is_valid_token 0, or a request index
 * outside [0, num_reqs)) is all -1 with lens 0.  The call passes no
 * replay_start, so none bounds the window.
 */
void oracle_decode_swa_indices_and_lens(
    const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* token_to_req, int32_t num_reqs, int64_t num_tokens,
    const int32_t* block_table, int64_t bt_stride, int32_t bt_width,
    const int32_t* base_offsets, int32_t block_size, int32_t window,
    const uint8_t* is_valid_token, int32_t* indices, int64_t out_stride,
    int32_t* lens) {
    for (int64_t t = 0; t < num_tokens; ++t) {
        int32_t* row = indices + t * out_stride;
        const int32_t r = token_to_req[t];
        const int ok = (is_valid_token ? is_valid_token[t] != 0 : 1) &&
                       r >= 0 && r < num_reqs;
        int32_t count = 0;
        if (!ok) {
            for (int32_t c = 0; c < window; ++c) row[c] = -1;
            lens[t] = 0;
            continue;
        }
        const int64_t qstart = query_start_loc[r];
        const int64_t qlen = (int64_t)query_start_loc[r + 1] - qstart;
        const int64_t pos = (int64_t)seq_lens[r] - qlen + (t - qstart);
        int64_t lo = pos - window + 1;
        if (lo < 0) lo = 0;
        const int32_t* trow = block_table + (int64_t)r * bt_stride;
        const int64_t base = base_offsets ? base_offsets[r] : 0;
        for (int32_t c = 0; c < window; ++c) {
            const int64_t p = lo + c;
            const int32_t v = p <= pos ? slot_of(trow, bt_width, base, block_size, p) : -1;
            row[c] = v;
            if (v >= 0) ++count;
        }
        lens[t] = count;
    }
}

/*
 * [BE] _decode_compressed_attention_indices_and_lens for a compress ratio other
 * than 4 (printed in full): token t of request r at positions[t] sees
 * n = clamp(floor((positions[t] + 1) / ratio), 0, width) compressed entries;
 * column j < width holds the slot of compressed entry j through the compressed
 * table row (logical page j / bs minus the request's base logical page) when
 * j < n and that page exists, else -1; lens[t] = n -- the count of visible
 * entries, including any whose page is missing, as printed -- and 0 for a
 * padding token (is_valid_token 0; and, a reading shared with the other
 * builders, a request index outside [0, num_reqs), whose row is all -1).
 * Slots beyond INT32_MAX are -1 (the builders' common reading).
 */
void oracle_compute_dense_compressed_indices_and_lens(
    const int64_t* positions, int64_t num_tokens, const int32_t* token_to_req,
    int32_t num_reqs, const int32_t* block_table, int64_t bt_stride,
    int32_t bt_width, const int32_t* base_offsets, int32_t block_size,
    int32_t compress_ratio, int32_t width, const uint8_t* is_valid_token,
    int32_t* indices, int64_t out_stride, int32_t* lens) {
    for (int64_t t = 0; t < num_tokens; ++t) {
        int32_t* row = indices + t * out_stride;
        const int32_t r = token_to_req[t];
        const int ok = (is_valid_token ? is_valid_token[t] != 0 : 1) &&
                       r >= 0 && r < num_reqs;
        if (!ok) {
            for (int32_t j = 0; j < width; ++j) row[j] = -1;
            lens[t] = 0;
            continue;
        }
        /* floor division of pos + 1 by the ratio, then the clamp to [0, width] */
        const int64_t num = positions[t] + 1;
        int64_t n = num >= 0 ? num / compress_ratio
                             : -((-num + compress_ratio - 1) / compress_ratio);
        if (n < 0) n = 0;
        if (n > width) n = width;
        const int32_t* trow = block_table + (int64_t)r * bt_stride;
        const int64_t base = base_offsets ? base_offsets[r] : 0;
        for (int32_t j = 0; j < width; ++j)
            row[j] = j < n ? slot_of(trow, bt_width, base, block_size, j) : -1;
        lens[t] = (int32_t)n;
    }
}

/*
 * [OPS] deepseek_v4_build_dense_prefill_local_compressed_indices(positions,
 * compress_ratio, width, out) as [BE] _dense_prefill_local_compressed_indices
 * calls it on the HCA prefill workspace path: the body is not printed; read as
 * the request-local form of the dense decode rule, out[t][j] = j for
 * j < min(floor((positions[t] + 1) / ratio), width), else -1.  The rows are the
 * top-k input of the workspace-relative combine.
 */
void oracle_build_dense_prefill_local_compressed_indices(
    const int64_t* positions, int64_t num_tokens, int32_t compress_ratio,
    int32_t width, int32_t* out, int64_t out_stride) {
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t num = positions[t] + 1;
        int64_t n = num >= 0 ? num / compress_ratio
                             : -((-num + compress_ratio - 1) / compress_ratio);
        if (n < 0) n = 0;
        if (n > width) n = width;
        for (int32_t j = 0; j < width; ++j) out[t * out_stride + j] = j < n ? j : -1;
    }
}

/*
 * [OPS] deepseek_v4_combine_dense_swa_indices as [BE] _prefill_workspace calls
 * it for layers without a compressed cache (compress_ratio <= 1, where the
 * compressed lengths are all zero and compressed_base is 0); the body is not
 * printed.  Read as the window columns of the workspace-relative combine with
 * the token's position given: column c < window holds position
 * p = lo + c, lo = max(positions[t] - window + 1, 0), as workspace row
 * r * workspace_width + compressed_base + (p - g0) when g0 <= p <= positions[t],
 * g0 = seq_lens[r] - gather_lens[r], else -1 (rows beyond INT32_MAX: -1);
 * lens = entries >= 0; a request index outside [0, num_reqs) gives an all -1
 * row with lens 0.
 */
void oracle_combine_dense_swa_indices(
    const int64_t* positions, const int32_t* token_to_req,
    const int32_t* seq_lens, const int32_t* gather_lens, int32_t num_reqs,
    int64_t num_tokens, int32_t window, int64_t workspace_width,
    int64_t compressed_base, int32_t* indices, int64_t out_stride,
    int32_t* lens) {
    for (int64_t t = 0; t < num_tokens; ++t) {
        int32_t* row = indices + t * out_stride;
        const int32_t r = token_to_req[t];
        if (r < 0 || r >= num_reqs) {
            for (int32_t c = 0; c < window; ++c) row[c] = -1;
            lens[t] = 0;
            continue;
        }
        const int64_t pos = positions[t];
        const int64_t g0 = (int64_t)seq_lens[r] - gather_lens[r];
        const int64_t rbase = (int64_t)r * workspace_width;
        int64_t lo = pos - window + 1;
        if (lo < 0) lo = 0;
        int32_t count = 0;
        for (int32_t c = 0; c < window; ++c) {
            const int64_t p = lo + c;
            int64_t v = -1;
            if (p <= pos && p >= g0) v = rbase + compressed_base + (p - g0);
            if (v > INT32_MAX) v = -1;
            row[c] = (int32_t)v;
            if (v >= 0) ++count;
        }
        lens[t] = count;
    }
}

/* ------------------------------------------------------------------------ */
/* Indexer-key variants: the FP8 indexer record and indexer_k_norm_rope_store */
/* ------------------------------------------------------------------------ */

/*
 * Per-row FP8 quantization with one power-of-two binary32 scale ([OPS]
 * _fp8_e4m3_pow2_bytes and _write_deepseek_v4_indexer_fp8_cache_capturable):
 * scale = 2^ceil(log2(max(amax / 448, 1e-10))) -- the quotient is floored, not
 * amax; the ceiling is taken exactly on the binary32 quotient, as for the
 * UE8M0 record -- and code = e4m3(clamp(x / scale, -448, 448)).  Returns the
 * scale.
 */
static float fp8_pow2_row(const float* x, int32_t n, uint8_t* codes) {
    float amax = 0.0f;
    for (int32_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float q = amax / 448.0f;
    if (q < 1.0e-10f) q = 1.0e-10f;
    const float scale = pow2f(oracle_ceil_log2(q));
    for (int32_t i = 0; i < n; ++i) {
        float v = x[i] / scale;
        if (v > 448.0f) v = 448.0f;
        if (v < -448.0f) v = -448.0f;
        codes[i] = oracle_e4m3_encode(v);
    }
    return scale;
}

/*
 * Per-32-block MXFP4 quantization of binary32 values, the rule of
 * oracle_write_indexer_mxfp4_cache: e = ceil(log2(max(amax, 1e-4) / 6)), scale
 * byte clamp(e + 127, 0, 254), code = e2m1(x * 2^-e), even element in the low
 * nibble.
 */
static void mxfp4_row(const float* x, int32_t n, uint8_t* vals, uint8_t* scl) {
    for (int32_t b = 0; b < n / 32; ++b) {
        float amax = 0.0f;
        for (int j = 0; j < 32; ++j) {
            float a = fabsf(x[b * 32 + j]);
            if (a > amax) amax = a;
        }
        float a = (amax < 1.0e-4f) ? 1.0e-4f : amax;
        int32_t e = oracle_ceil_log2(a / 6.0f);
        int32_t byte = e + 127;
        if (byte < 0) byte = 0;
        if (byte > 254) byte = 254;
        scl[b] = (uint8_t)byte;
        float p = pow2f(-e);
        for (int j = 0; j < 32; j += 2) {
            uint8_t lo = oracle_e2m1_encode(x[b * 32 + j] * p);
            uint8_t hi = oracle_e2m1_encode(x[b * 32 + j + 1] * p);
            vals[(b * 32 + j) / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/*
 * [OPS] write_deepseek_v4_indexer_fp8_cache: FP8 indexer keys in the
 * "[values | fp32 scale]" page layout.  Page: [block_size x head_dim e4m3
 * bytes][block_size x 4-byte little-endian binary32 scales]; token off of a
 * page at off * head_dim and block_size * head_dim + off * 4.  Slots < 0 are
 * skipped; slots >= capacity are skipped and counted (returned).
 */
int64_t oracle_write_indexer_fp8_cache(
    const uint16_t* k, int64_t k_row_stride, const int64_t* slot_mapping,
    int64_t num_tokens, uint8_t* cache, int64_t num_pages,
    int64_t page_stride, int32_t block_size, int32_t head_dim) {
    const int64_t capacity = num_pages * (int64_t)block_size;
    int64_t errors = 0;
    float x[1024];
    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t s = slot_mapping[i];
        if (s < 0) continue;
        if (s >= capacity) {
            ++errors;
            continue;
        }
        const int64_t page = s / block_size, off = s % block_size;
        uint8_t* base = cache + page * page_stride;
        for (int32_t d = 0; d < head_dim; ++d) x[d] = oracle_bf16_to_f32(k[i * k_row_stride + d]);
        const float scale = fp8_pow2_row(x, head_dim, base + off * head_dim);
        memcpy(base + (int64_t)block_size * head_dim + off * 4, &scale, 4);
    }
    return errors;
}

/* Pairwise (recursive halving) binary32 sum of v[0..n), n a power of two. */
static float pairwise_sum(const float* v, int32_t n) {
    if (n == 1) return v[0];
    return pairwise_sum(v, n / 2) + pairwise_sum(v + n / 2, n / 2);
}

/*
 * [VLLM] indexer_k_norm_rope_store(k_pre, positions, cos_sin_cache,
 * rms_norm_weight, rms_norm_eps, k_cache, kv_slot_mapping, compress_ratio,
 * use_fp4_cache): k_norm -> RoPE -> quant -> paged store of 128-dim indexer
 * keys (64 RoPE dims).  The kernel is not printed; the stages follow the
 * pages' torch forms of the same steps:
 *   emission: token t writes a key when kv_slot_mapping[t] >= 0 and it closes
 *     its compress group, (positions[t] + 1) % ratio == 0 (the valid_token rule
 *     of [OPS] _compress_v4_state_windows_capturable; "only group-boundary rows
 *     are read");
 *   RMSNorm ([OPS] _compress_v4_state_windows_capturable), binary32:
 *     variance = (sum of x_d * x_d) / 128 with the sum taken pairwise
 *     (recursive halving in index order -- a reading: no order is printed);
 *     r = 1 / sqrt(variance + eps) as an IEEE binary32 square root followed
 *     by an IEEE binary32 division (a reading: the printed rsqrt is a binary32
 *     library call of unstated accuracy); y_d = (x_d * r) * weight_d;
 *   RoPE ([OPS] _apply_gptj_rope_tail_rows, GPT-J pairs on the last 64 dims):
 *     for i < 32, e = y[64 + 2i], o = y[65 + 2i], c = cs[p][i], s = cs[p][32 + i]:
 *     y[64 + 2i] = e*c - o*s, y[65 + 2i] = e*s + o*c (each product and sum
 *     rounded to binary32), at the group's first position
 *     p = floor(positions[t] / ratio) * ratio (the compressed_positions of
 *     [OPS] deepseek_v4_csa_indexer_cache_insert);
 *   quant + store: record 1 = the MXFP4 record, record 2 = the FP8 indexer
 *     record, at kv_slot_mapping[t].
 * Slots >= capacity and RoPE rows p outside [0, max_pos) are skipped and
 * counted (returned).
 */
int64_t oracle_indexer_k_norm_rope_store(
    const uint16_t* k_pre, int64_t k_row_stride, const int64_t* positions,
    const float* cos_sin_cache, int64_t cs_stride, int64_t max_pos,
    const float* rms_norm_weight, float rms_norm_eps,
    const int64_t* slot_mapping, int64_t num_tokens, int32_t compress_ratio,
    int32_t record, uint8_t* cache, int64_t num_pages, int64_t page_stride,
    int32_t block_size) {
    const int32_t D = 128, R = 64, nope = D - R;
    const int64_t capacity = num_pages * (int64_t)block_size;
    int64_t errors = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t s = slot_mapping[t];
        if (s < 0) continue;
        const int64_t pos = positions[t];
        /* group boundary: (pos + 1) mod ratio == 0 (floor modulus) */
        int64_t m = (pos + 1) % compress_ratio;
        if (m < 0) m += compress_ratio;
        if (m != 0) continue;
        /* floor(pos / ratio) * ratio */
        int64_t q = pos / compress_ratio;
        if (pos % compress_ratio != 0 && pos < 0) q -= 1;
        const int64_t p = q * compress_ratio;
        if (s >= capacity || p < 0 || p >= max_pos) {
            ++errors;
            continue;
        }
        float x[128], sq[128], y[128];
        for (int32_t d = 0; d < D; ++d) {
            x[d] = oracle_bf16_to_f32(k_pre[t * k_row_stride + d]);
            sq[d] = x[d] * x[d];
        }
        const float variance = pairwise_sum(sq, D) / 128.0f;
        const float r = 1.0f / sqrtf(variance + rms_norm_eps);
        for (int32_t d = 0; d < D; ++d) y[d] = (x[d] * r) * rms_norm_weight[d];
        const float* cs = cos_sin_cache + p * cs_stride;
        for (int32_t i = 0; i < R / 2; ++i) {
            const float e = y[nope + 2 * i], o = y[nope + 2 * i + 1];
            const float c = cs[i], sn = cs[R / 2 + i];
            const float ec = e * c, os = o * sn, es = e * sn, oc = o * c;
            y[nope + 2 * i] = ec - os;
            y[nope + 2 * i + 1] = es + oc;
        }
        const int64_t page = s / block_size, off = s % block_size;
        uint8_t* base = cache + page * page_stride;
        if (record == 1) {
            mxfp4_row(y, D, base + off * (D / 2), base + (int64_t)block_size * (D / 2) + off * (D / 32));
        } else {
            const float scale = fp8_pow2_row(y, D, base + off * D);
            memcpy(base + (int64_t)block_size * D + off * 4, &scale, 4);
        }
    }
    return errors;
}

/* ------------------------------------------------------------------------ */
/* Compressed-KV producer: compressor state, window pooling, record insert   */
/* ------------------------------------------------------------------------ */

/*
 * exp of a binary32, by Cody and Waite's argument reduction (Cody & Waite,
 * "Software Manual for the Elementary Functions", 1980) and the Taylor series:
 *   k = nearest integer to x / ln 2 (x * 1.44269504, rounded to even);
 *   r = x - k*ln2_hi - k*ln2_lo with ln2_hi = 0.693145751953125 (16 significant
 *       bits, so k*ln2_hi is exact for |k| <= 256) and ln2_lo = ln 2 - ln2_hi,
 *       each step one fused multiply-add;
 *   exp(r) = 1 + r + r^2/2! + ... + r^7/7! by Horner with fused multiply-adds
 *       (|r| <= 0.347: the first omitted term is below 6e-9 relative);
 *   result = p * 2^k, as one multiply by a normal power of two (two when 2^k
 *       is not normal, so a subnormal result is rounded once).
 * Every operation is an IEEE binary32 one, so the kernels evaluate the same
 * sequence to the same bits.  Pinned against the C library's exp within 2 ulp.
 */
float oracle_exp_cw(float x) {
    if (isnan(x)) return x;
    if (x > 88.7228f) return INFINITY;
    if (x < -103.98f) return 0.0f;
    const float k = rintf(x * 1.44269504f);
    float r = fmaf(-k, 0.693145751953125f, x);
    r = fmaf(-k, 1.42860677e-06f, r);
    float p = 1.98412698e-04f;            /* 1/7! */
    p = fmaf(p, r, 1.38888889e-03f);      /* 1/6! */
    p = fmaf(p, r, 8.33333333e-03f);      /* 1/5! */
    p = fmaf(p, r, 4.16666667e-02f);      /* 1/4! */
    p = fmaf(p, r, 1.66666667e-01f);      /* 1/3! */
    p = fmaf(p, r, 0.5f);                 /* 1/2! */
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    const int ki = (int)k;
    if (ki < -126) return (p * pow2f(ki + 64)) * pow2f(-64);
    if (ki > 127) return (p * pow2f(ki - 1)) * 2.0f;
    return p * pow2f(ki);
}

/*
 * [OPS] save_deepseek_v4_compressor_state: the compressor's residual state of
 * each token, [kv_state | score_state] (each state_width binary32 values), in a
 * paged cache [pages, block_size, 2 * state_width] at the token's state slot;
 * the score state "includes the APE row selected by position % compress_ratio".
 * The kernel is not printed; read as state[slot] = [kv[t], score[t] + ape[pos %
 * ratio]] (binary32 adds).  Slots < 0 are skipped; slots beyond the cache are
 * skipped and counted.
 */
int64_t oracle_save_compressor_state(
    const float* kv, const float* score, int64_t in_stride, const float* ape,
    int32_t state_width, const int64_t* slot_mapping, const int64_t* positions,
    int64_t num_tokens, int32_t compress_ratio, float* state_cache, int64_t num_pages,
    int32_t block_size) {
    const int64_t capacity = num_pages * (int64_t)block_size;
    int64_t errors = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t s = slot_mapping[t];
        if (s < 0) continue;
        if (s >= capacity) {
            ++errors;
            continue;
        }
        int64_t a = positions[t] % compress_ratio;
        if (a < 0) a += compress_ratio;
        float* row = state_cache + s * 2 * (int64_t)state_width;
        for (int32_t d = 0; d < state_width; ++d) {
            row[d] = kv[t * in_stride + d];
            row[state_width + d] = score[t * in_stride + d] + ape[a * state_width + d];
        }
    }
    return errors;
}

/*
 * [OPS] deepseek_v4_csa_compress_kv_cache_insert (compress_ratio 4, overlap) and
 * deepseek_v4_hca_compress_kv_cache_insert (128, no overlap), whose torch form is
 * _compress_v4_state_windows_capturable then _write_fp8_ds_mla_cache_rows_capturable
 * (_fp8_ds_mla_cache_rows):
 *   emission: token t writes when its state slot and kv_slot_mapping[t] are >= 0
 *     and (pos + 1) % ratio == 0;
 *   window: the window = (overlap ? 2 : 1) * ratio positions pos - window + 1 + j;
 *     position p is present when p >= 0, its logical page floor(p / bs) - base[r]
 *     lies in [0, width) and the table entry is >= 0; its state row is
 *     state[entry * bs + p % bs];
 *   head_dim values per row: the kv slice and the score slice at column offset
 *     head_dim for j >= ratio under overlap (the newer positions take the second
 *     slice), else 0;
 *   pooling per column d: scores of absent positions are -1e30 and their kv 0;
 *     m = max_j s_j; e_j = exp(s_j - m); sum = e_0 + e_1 + ... (ascending j);
 *     w_j = e_j / sum; c_d = kv_0 w_0 + kv_1 w_1 + ... (ascending j; each product
 *     and sum rounded) -- the order is a reading (none is printed); exp is
 *     oracle_exp_cw;
 *   RMSNorm as indexer_k_norm_rope_store's (pairwise sum of squares / head_dim,
 *     IEEE sqrt then division, (c * r) * weight);
 *   record: the fp8_ds_mla insert of the bf16 row [bf16(normed) on the nope dims |
 *     bf16(GPT-J RoPE of the binary32 normed tail at floor(pos / ratio) * ratio)],
 *     i.e. oracle_quantize_and_insert_k_cache's UE8M0 rule (as
 *     _fp8_ds_mla_cache_rows quantises normed.to(bf16)).
 * Slots beyond a cache and RoPE rows outside [0, max_pos) are skipped and counted.
 */
int64_t oracle_compress_kv_cache_insert(
    const float* state_cache, int64_t state_num_pages, int32_t state_block_size,
    int32_t state_width, const int32_t* token_to_req, const int64_t* positions,
    const int64_t* state_slot_mapping, const int32_t* block_table, int64_t bt_stride,
    int32_t bt_width, const int32_t* base_offsets, int32_t num_reqs, int64_t num_tokens,
    int32_t compress_ratio, int32_t overlap, int32_t head_dim, int32_t rope_dim,
    const float* rms_norm_weight, float rms_norm_eps, const float* cos_sin_cache,
    int64_t cs_stride, int64_t max_pos, uint8_t* kv_cache, int64_t kv_num_pages,
    int64_t kv_page_stride, int32_t kv_block_size, const int64_t* kv_slot_mapping) {
    const int32_t window = (overlap ? 2 : 1) * compress_ratio;
    const int64_t state_cap = state_num_pages * (int64_t)state_block_size;
    const int64_t kv_cap = kv_num_pages * (int64_t)kv_block_size;
    const int32_t nope = head_dim - rope_dim;
    int64_t errors = 0;
    float c[1024], sq[1024], y[1024];
    int64_t rowidx[256];
    uint16_t bf[1024];
    for (int64_t t = 0; t < num_tokens; ++t) {
        if (state_slot_mapping[t] < 0 || kv_slot_mapping[t] < 0) continue;
        const int64_t pos = positions[t];
        int64_t m = (pos + 1) % compress_ratio;
        if (m < 0) m += compress_ratio;
        if (m != 0) continue;
        int64_t q = pos / compress_ratio;
        if (pos % compress_ratio != 0 && pos < 0) q -= 1;
        const int64_t prow = q * compress_ratio;
        const int32_t r = token_to_req[t];
        if (kv_slot_mapping[t] >= kv_cap || prow < 0 || prow >= max_pos || r < 0 ||
            r >= num_reqs) {
            ++errors;
            continue;
        }
        /* the window's state rows (-1: absent) */
        const int64_t base = base_offsets ? base_offsets[r] : 0;
        for (int32_t j = 0; j < window; ++j) {
            const int64_t p = pos - window + 1 + j;
            rowidx[j] = -1;
            if (p < 0) continue;
            const int64_t lp = p / state_block_size - base;
            if (lp < 0 || lp >= bt_width) continue;
            const int32_t entry = block_table[(int64_t)r * bt_stride + lp];
            if (entry < 0) continue;
            const int64_t srow = (int64_t)entry * state_block_size + p % state_block_size;
            if (srow >= state_cap) continue;
            rowidx[j] = srow;
        }
        /* softmax pooling per column */
        for (int32_t d = 0; d < head_dim; ++d) {
            float s[256], kvv[256];
            for (int32_t j = 0; j < window; ++j) {
                const int32_t off = (overlap && j >= compress_ratio) ? head_dim : 0;
                if (rowidx[j] < 0) {
                    s[j] = -1.0e30f;
                    kvv[j] = 0.0f;
                } else {
                    const float* row = state_cache + rowidx[j] * 2 * (int64_t)state_width;
                    kvv[j] = row[off + d];
                    s[j] = row[state_width + off + d];
                }
            }
            float mx = s[0];
            for (int32_t j = 1; j < window; ++j)
                if (s[j] > mx) mx = s[j];
            float sum = 0.0f;
            for (int32_t j = 0; j < window; ++j) sum = sum + oracle_exp_cw(s[j] - mx);
            float acc = 0.0f;
            for (int32_t j = 0; j < window; ++j) {
                const float w = oracle_exp_cw(s[j] - mx) / sum;
                acc = acc + kvv[j] * w;
            }
            c[d] = acc;
        }
        /* RMSNorm */
        for (int32_t d = 0; d < head_dim; ++d) sq[d] = c[d] * c[d];
        const float variance = pairwise_sum(sq, head_dim) / (float)head_dim;
        const float rr = 1.0f / sqrtf(variance + rms_norm_eps);
        for (int32_t d = 0; d < head_dim; ++d) y[d] = (c[d] * rr) * rms_norm_weight[d];
        /* bf16 row: the nope dims rounded as they are, the tail after GPT-J RoPE */
        for (int32_t d = 0; d < nope; ++d) bf[d] = oracle_bf16_from_f32(y[d]);
        const float* cs = cos_sin_cache + prow * cs_stride;
        for (int32_t i = 0; i < rope_dim / 2; ++i) {
            const float e = y[nope + 2 * i], o = y[nope + 2 * i + 1];
            const float cc = cs[i], sn = cs[rope_dim / 2 + i];
            const float ec = e * cc, os = o * sn, es = e * sn, oc = o * cc;
            bf[nope + 2 * i] = oracle_bf16_from_f32(ec - os);
            bf[nope + 2 * i + 1] = oracle_bf16_from_f32(es + oc);
        }
        errors += oracle_quantize_and_insert_k_cache(bf, head_dim, kv_slot_mapping + t, 1,
                                                     kv_cache, kv_num_pages, kv_page_stride,
                                                     kv_block_size, head_dim, rope_dim, 1);
    }
    return errors;
}

void oracle_exp_cw_array(const float* x, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_exp_cw(x[i]);
}
