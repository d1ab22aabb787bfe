/*
 * oracle.h -- plain CPU reference of the DeepSeek-Sparse-Attention lightning-indexer
 * hot path (K store, Q quant, paged MQA logits, per-query top-k).
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this library. It shares no code, header, table or helper with the CUDA
 * library under sparse_attention_indexer_mqa_gb300/csrc; both follow the same written
 * rules, stated per function in oracle.c.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] vllm PR 57517 "[ROCm][Perf] Add AITER paged MXFP4 sparse indexing on gfx950"
 *   [P2] vllm PR 60834 (MXFP4 indexer for DeepSeek-V4: K write, Q quant, scoring)
 *   [P3] vllm PR 53094 "[ROCm][Perf] Fuse DSA indexer QK preprocessing with AITER"
 *
 * Conventions: bf16 values travel as uint16 bit patterns; every buffer is host memory
 * owned by the caller; nothing here allocates memory that outlives a call.
 */
#ifndef IDX_ORACLE_H
#define IDX_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype / rope codes (same numeric values as the public ABI, restated here). */
#define ORC_MXFP4 0
#define ORC_FP8 1
#define ORC_ROPE_NONE 0
#define ORC_ROPE_NEOX 1
#define ORC_ROPE_INTERLEAVED 2

/* --- element encoders -------------------------------------------------------------- */
uint8_t orc_e2m1_encode(float v);          /* nearest e2m1, ties to even code, sat. +-6 */
double orc_e2m1_decode(uint8_t code);      /* low nibble only */
uint8_t orc_e4m3_encode(float v);          /* nearest e4m3fn, ties to even, sat. +-448 */
double orc_e4m3_decode(uint8_t code);
int orc_mx_shared_exponent(float amax);    /* floor(log2 amax) - 2, clamped, amax==0 -> -127 */
/* element-wise over arrays (for sweeps) */
void orc_e2m1_encode_n(const float* v, int64_t n, uint8_t* out);
void orc_e4m3_encode_n(const float* v, int64_t n, uint8_t* out);

/* --- row steps ---------------------------------------------------------------------- */
void orc_layernorm128(const float* x, const float* gamma, const float* beta, float eps,
                      float* y);
void orc_rope128(float* x, const float* cos_sin_row, int mode);
void orc_mxfp4_quant128(const float* x, uint8_t* codes64, uint8_t* scales4);
void orc_fp8_quant128(const float* x, uint8_t* codes128, float* scale);

/* --- page layout (per token, per page size) --------------------------------------- */
int64_t orc_page_bytes(int dtype, int page_size);
/* byte offset inside a page of the code byte holding packed element pair j (MXFP4,
 * j in 0..63) or element j (FP8, j in 0..127) of in-page token s */
int64_t orc_code_offset(int dtype, int page_size, int s, int j);
/* byte offset of scale byte b (MXFP4, b in 0..3) or of the fp32 scale (FP8, b ignored) */
int64_t orc_scale_offset(int dtype, int page_size, int s, int b);

/* --- whole steps -------------------------------------------------------------------- */
int orc_k_store(const uint16_t* k, int64_t n_rows, int64_t k_row_stride,
                const int64_t* slot_mapping, const int32_t* positions,
                const float* cos_sin, int32_t max_pos, int rope, int apply_norm,
                const float* gamma, const float* beta, float eps, int dtype,
                uint8_t* pool, int64_t num_pages, int32_t page_size, int64_t page_stride);

/* compressor front end (see oracle.c, readings R13-R16) */
float orc_exp_neg(float a);
void orc_rmsnorm128(const float* x, const float* gamma, float eps, float* y);
void orc_compress_pool128(const uint16_t* k_raw, const uint16_t* gate, int64_t row_stride,
                          int64_t lo, int64_t hi, float* out);
int orc_compress_k_store(const uint16_t* k_raw, const uint16_t* gate, int64_t n_raw, int64_t row_stride,
                         const int64_t* boundary, const int64_t* first, int64_t n_entries,
                         int32_t ratio, const int64_t* slot_mapping, const int32_t* positions,
                         const float* cos_sin, int32_t max_pos, int rope, int norm,
                         const float* gamma, const float* beta, float eps, int dtype,
                         uint8_t* pool, int64_t num_pages, int32_t page_size,
                         int64_t page_stride);

int orc_q_quant(const uint16_t* q, int64_t T, int32_t H, const int32_t* positions,
                const float* cos_sin, int32_t max_pos, int rope, const float* w_in,
                float softmax_scale, float head_scale, int dtype, uint8_t* q_codes,
                uint8_t* q_scales, float* w_out);

/* visible key count of query t (returns -1 if t is outside every sequence) */
int64_t orc_visible(int64_t t, const int32_t* seq_lens_k, const int32_t* cu_seqlens_q,
                    int32_t B, int causal);

/* logits for the query rows listed in rows[0..n_rows) (all rows if rows == NULL, then
 * n_rows = T); out is double [n_rows][ld]; entries past visible(t) are left as is. */
int orc_mqa_logits(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                   int64_t T, int32_t H, int dtype, const uint8_t* pool, int64_t num_pages,
                   int32_t page_size, int64_t page_stride, const int32_t* page_table,
                   int32_t pt_stride, const int32_t* seq_lens_k, const int32_t* cu_seqlens_q,
                   int32_t B, int causal, const int64_t* rows, int64_t n_rows, double* out,
                   int64_t ld, int n_threads);

/* top-k over double logits rows [n_rows][ld]; row r belongs to query rows[r] (or r) */
int orc_topk(const double* logits, int64_t ld, const int32_t* seq_lens_k,
             const int32_t* cu_seqlens_q, int32_t B, int causal, const int64_t* rows,
             int64_t n_rows, int32_t k, int32_t* out_idx, int n_threads);

/* candidate-pool top-k (see oracle.c, reading R17) */
int orc_topk_cand(const double* logits, int64_t ld, const int32_t* seq_lens_k,
                  const int32_t* cu_seqlens_q, int32_t B, int causal, const int64_t* rows,
                  int64_t n_rows, const int32_t* cand, int32_t cand_stride, const int32_t* n_cand,
                  int32_t page_size, int32_t k, int32_t* out_idx, int n_threads);

#ifdef __cplusplus
}
#endif

#endif
