/*
 * idx.h -- C ABI of the GB300 (sm_103a) DeepSeek-Sparse-Attention lightning-indexer
 * hot path: K store, Q quant, paged MQA-logits scorer, per-query top-k.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] vllm PR 57517 "[ROCm][Perf] Add AITER paged MXFP4 sparse indexing on gfx950"
 *   [P2] vllm PR 60834 (MXFP4 indexer for DeepSeek-V4: K write, Q quant, scoring)
 *   [P3] vllm PR 53094 "[ROCm][Perf] Fuse DSA indexer QK preprocessing with AITER"
 *
 * Common rules for every entry point
 *   Ownership. The caller allocates and owns every buffer (device memory unless stated)
 *     and the stream. The library never allocates, frees or synchronises; every call only
 *     enqueues work on `stream` (NULL = the legacy default stream) and returns.
 *   Errors. Problems visible on the host (bad enum, unsupported size, NULL or misaligned
 *     pointer) return IDX_EINVAL / IDX_EUNSUPPORTED before anything is launched. A failed
 *     launch returns IDX_ECUDA. Data-dependent problems found on the device (a slot, page
 *     id or position out of range, a bounded wait that ran out) never trap: the kernel
 *     skips the affected row or tile and ORs a bit into *dev_status, when dev_status is
 *     non-NULL (a device int32 the caller zeroes). See IDX_STATUS_* below.
 *   Vectors. D (head dim) is 128 and the rotary part is dims 0..63 ([P3] "Purpose": the
 *     fused path requires index_head_dim == 128 and qk_rope_head_dim == 64).
 *   bf16 inputs are passed as raw 16-bit patterns (uint16_t).
 */
#ifndef IDX_H
#define IDX_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    IDX_OK = 0,
    IDX_EINVAL = -1,       /* bad argument: NULL, misaligned, negative size, bad enum */
    IDX_EUNSUPPORTED = -2, /* valid but not implemented (page size, head count, k) */
    IDX_ECUDA = -3         /* a CUDA launch or attribute call failed */
} idx_status;

typedef enum { IDX_MXFP4 = 0, IDX_FP8 = 1 } idx_dtype;

typedef enum { IDX_ROPE_NONE = 0, IDX_ROPE_NEOX = 1, IDX_ROPE_INTERLEAVED = 2 } idx_rope;

/* bits ORed into *dev_status by the kernels */
#define IDX_STATUS_BAD_SLOT 0x1     /* slot >= num_pages * page_size: row skipped */
#define IDX_STATUS_BAD_POS 0x2      /* position outside [0, max_pos): row skipped */
#define IDX_STATUS_BAD_PAGE 0x4     /* page-table entry outside [0, num_pages): tile skipped */
#define IDX_STATUS_TIMEOUT 0x8      /* a bounded wait ran out: the CTA stopped early */
#define IDX_STATUS_BAD_LEN 0x10     /* a sequence's key or query count broke its bound: skipped */

/*
 * Page layout of the paged indexer K cache. This library owns it: callers learn it only
 * from idx_cache_layout, as the pages' integration reads the layout from a single owner
 * ([P2] "Changes / K write": the layout is read from one place only).
 *
 * MXFP4, 68 bytes per token ([P2] "Purpose": 68 B per token instead of 132 B for FP8):
 *   a page of P tokens is [64*P bytes of e2m1 codes][4*P bytes of E8M0 scales].
 *   Token s's 128 elements form four scale blocks of 32; block c is one 16-byte chunk
 *   whose byte i holds elements 32c+2i (low nibble) and 32c+2i+1 (high nibble).
 *   P = 128: chunk (s, c) at ((s/8)*4 + c)*128 + (s%8)*16;
 *            scale (s, c) at 8192 + (s%32)*16 + (s/32)*4 + c.
 *   P =  64: chunk (s, c) at (s/16)*1024 + ((s/8)%2)*512 + c*128 + (s%8)*16;
 *            scale (s, c) at 4096 + (s%16)*16 + (s/16)*4 + c.
 *   The chunk order is the K-major, unswizzled core-matrix order (8 rows x 16 bytes) of a
 *   128-row tcgen05 operand tile; the scale order is the tensor-memory scale-factor order.
 *   A P = 128 page is one tile; two P = 64 pages interleave into one tile. So a page is
 *   copied to shared memory as is and fed to the tensor core without a register pass:
 *   the analogue of the pages' "preshuffled page order" ([P2] "Purpose").
 * FP8, 132 bytes per token: a page is [128*P bytes of e4m3][P fp32 scales];
 *   element j of token s at (s/8)*1024 + (j/16)*128 + (s%8)*16 + j%16;
 *   the scale of token s at 128*P + 4*s.
 * Every page starts on a 16-byte boundary (page_stride % 16 == 0).
 */
typedef struct {
    int64_t page_bytes;      /* bytes of one page (68*P or 132*P) */
    int64_t code_offset;     /* offset of the code region in a page (0) */
    int64_t code_bytes;      /* 64*P or 128*P */
    int64_t scale_offset;    /* offset of the scale region (= code_bytes) */
    int64_t scale_bytes;     /* 4*P */
    int32_t bytes_per_token; /* 68 or 132 */
    int32_t page_size;       /* P */
} idx_layout;

/* Page size P must be 64 or 128 ([P1] "Performance and accuracy": --block-size 128;
 * [P2] "Scoring and metadata": 64-entry pages at compress ratio 4). Host-only call. */
int idx_cache_layout(int32_t dtype, int32_t page_size, idx_layout* out);

/*
 * K store ([P3] "Purpose" steps 1, 2 and 5; [P2] "Changes / K write"):
 * for each row r < n_rows of k (bf16, row r at k + r*k_row_stride, 16-byte aligned):
 *   x = fp32(k[r]); if apply_norm: x = LayerNorm(x; gamma, beta, eps);
 *   if rope != NONE: rotate dims 0..63 at positions[r] with the table cos_sin;
 *   quantise to dtype and write the token's 68 or 132 bytes at slot = slot_mapping[r]
 *   (page slot / P of the pool, in-page token slot % P).
 * Arithmetic: fp32, every operation correctly rounded, no fused multiply-add, LayerNorm
 *   with biased variance, rstd = 1/sqrt(var+eps), sums over a fixed tree (16 groups of 8
 *   consecutive values, then xor-butterfly 8, 4, 2, 1); MXFP4 block exponent
 *   floor(log2 amax) - 2 clamped to [-127, 127] (amax = 0 gives -127), elements x*2^-E
 *   rounded to nearest-even e2m1 with saturation at 6 and the input's sign; FP8 scale
 *   max(amax, 1e-10)/448, elements x/scale rounded to nearest-even e4m3 saturating at 448.
 * cos_sin: fp32 [max_pos][64] = cos of the 32 frequencies, then sin of them; 16-byte
 * aligned (IDX_EINVAL otherwise).
 * gamma, beta: fp32 [128]; both may be NULL (meaning 1 and 0) when apply_norm != 0.
 * slot_mapping: int64 [n_rows]; slot < 0 skips the row ([P3] "Purpose": PAD_SLOT_ID).
 * positions: int32 [n_rows]; may be NULL when rope == IDX_ROPE_NONE.
 * pool: the paged cache base (16-byte aligned); page p starts at pool + p*page_stride,
 *   page_stride >= page bytes and a multiple of 16 ([P1] "Purpose": shared-pool page
 *   strides and 64-bit physical-page rebasing). All offsets are computed in 64 bits.
 */
int idx_k_store(const uint16_t* k, int64_t n_rows, int64_t k_row_stride,
                const int64_t* slot_mapping, const int32_t* positions,
                const float* cos_sin, int32_t max_pos, int32_t rope, int32_t apply_norm,
                const float* gamma, const float* beta, float eps, int32_t dtype, void* pool,
                int64_t num_pages, int32_t page_size, int64_t page_stride,
                int32_t* dev_status, cudaStream_t stream);

/*
 * Q quant ([P2] "Changes / Q quant"; [P3] "Purpose" steps 2-4):
 * q: bf16 [T][H][128] contiguous; positions: int32 [T] (NULL if rope == NONE);
 * w_in: fp32 [T][H]. For each (t, h): RoPE at positions[t], then quantisation.
 * Output layout (this library's own, the packed Q of [P1] "Purpose"): per query, the
 * quantised heads form a tensor-core operand image of Hq = roundup(H, 8) rows, K-major,
 * 8-row groups of 16-byte chunks, so the scorers copy it to shared memory unchanged.
 *   MXFP4: q_codes [T][Hq][64] bytes; chunk c (scale block c) of head h of query t at
 *            t*Hq*64 + ((h/8)*4 + c)*128 + (h%8)*16, byte i of the chunk holding elements
 *            32c+2i (low nibble) and 32c+2i+1 (high nibble);
 *          q_scales [T][512] bytes (16-byte aligned): the E8M0 scale of block c of head h at
 *            t*512 + (h%32)*16 + (h/32)*4 + c (the tensor-memory scale-factor order);
 *          w_out[t,h] = w_in[t,h] * c.
 *   FP8:   q_codes [T][Hq][128] e4m3; element j of head h at
 *            t*Hq*128 + ((h/8)*8 + j/16)*128 + (h%8)*16 + j%16 (one fp32 scale per
 *            128-element group, i.e. per (t, h));
 *          q_scales: optional fp32 [T][H] copy of those scales (may be NULL);
 *          w_out[t,h] = (w_in[t,h] * c) * scale[t,h]   (the q-scale fold, [P3] step 4).
 *   c = fp32(softmax_scale * head_scale), one rounding. Heads h in [H, Hq) are written as
 *   zero codes with scale bytes 127; the scale bytes of heads >= Hq are not written.
 * Same rounding rules as idx_k_store. H in 1..64.
 */
int idx_q_quant(const uint16_t* q, int64_t T, int32_t H, const int32_t* positions,
                const float* cos_sin, int32_t max_pos, int32_t rope, const float* w_in,
                float softmax_scale, float head_scale, int32_t dtype, uint8_t* q_codes,
                void* q_scales, float* w_out, int32_t* dev_status, cudaStream_t stream);

/*
 * Compressed K store, the DeepSeek-V4 indexer's K write ([P2] "Changes / K write": the
 * indexer K comes from its own compressor; one fused kernel pools the raw rows by
 * softmax-gated overlap pooling, applies RMSNorm, RoPE and the quantisation, and stores,
 * with nothing before the norm reaching memory; [P2] "Purpose": compress ratio 4, 64-entry
 * pages). One cache entry per boundary token:
 *   k_raw, gate: bf16 [n_raw][row_stride] (the first 128 of each row used), 16-byte aligned,
 *     row_stride >= 128 and a multiple of 8 (the two share the stride);
 *   boundary, first: int64 [n_entries]; entry e pools rows lo..hi with hi = boundary[e] and
 *     lo = max(first[e], hi - 2*ratio + 1) (its own ratio rows and the ratio rows before them,
 *     clipped at first[e], the first raw row of the entry's sequence);
 *   per dimension d: m = max of gate[i][d] over the window, w_i = exp(gate[i][d] - m),
 *     pooled[d] = (sum_i w_i * k_raw[i][d]) / (sum_i w_i), sums in row order;
 *   then norm (0 none, 1 LayerNorm as in idx_k_store, 2 RMSNorm:
 *     y = (x * (1 / sqrt(sum(x^2) / 128 + eps))) * gamma), RoPE at positions[e], the
 *     quantisation and the paged write at slot_mapping[e], all as in idx_k_store.
 * Arithmetic: fp32, the pooled row is not rounded to bf16; exp is Cody-Waite reduction plus a
 *   degree-7 Taylor polynomial in fused multiply-adds (<= 1 ulp on [-87, 0], 0 below -87);
 *   the sum of w_i * k_raw by fused multiply-adds, every other operation rounded once; the
 *   bytes are a function of the inputs alone (the launch shape does not change them).
 * ratio: 1..128 (IDX_EUNSUPPORTED otherwise). slot_mapping[e] < 0 skips the entry. An entry
 *   whose slot is past the pool sets IDX_STATUS_BAD_SLOT, whose window is not inside the raw
 *   rows (first[e] < 0, first[e] > boundary[e] or boundary[e] >= n_raw) sets
 *   IDX_STATUS_BAD_LEN, whose position is outside [0, max_pos) sets IDX_STATUS_BAD_POS; such
 *   entries are not written. Other arguments as in idx_k_store (gamma/beta may be NULL:
 *   1 and 0). Reads k_raw, gate and the index arrays; writes only the entries' slots.
 */
int idx_compress_k_store(const uint16_t* k_raw, const uint16_t* gate, int64_t n_raw, int64_t row_stride,
                         const int64_t* boundary, const int64_t* first, int64_t n_entries,
                         int32_t ratio, const int64_t* slot_mapping, const int32_t* positions,
                         const float* cos_sin, int32_t max_pos, int32_t rope, int32_t norm,
                         const float* gamma, const float* beta, float eps, int32_t dtype, void* pool,
                         int64_t num_pages, int32_t page_size, int64_t page_stride,
                         int32_t* dev_status, cudaStream_t stream);

/*
 * K store and Q quant in one launch ([P3] "Purpose": the indexer's QK pre-processing as a
 * single fused kernel instead of separate launches). Computes exactly what idx_k_store(k,
 * n_rows, k_row_stride, slot_mapping, k_positions, cos_sin, max_pos, k_rope, apply_norm,
 * gamma, beta, eps, dtype, pool, ...) followed by idx_q_quant(q, T, H, q_positions, cos_sin,
 * max_pos, q_rope, w_in, softmax_scale, head_scale, dtype, q_codes, q_scales, w_out) would,
 * with the same arguments, layouts, rounding, checks and status bits; the cache and the Q
 * image share one dtype and one RoPE table. Either half may be empty (n_rows = 0 or T = 0).
 */
int idx_qk_prep(const uint16_t* k, int64_t n_rows, int64_t k_row_stride, const int64_t* slot_mapping,
                const int32_t* k_positions, int32_t k_rope, int32_t apply_norm, const float* gamma,
                const float* beta, float eps, void* pool, int64_t num_pages, int32_t page_size,
                int64_t page_stride, const uint16_t* q, int64_t T, int32_t H,
                const int32_t* q_positions, int32_t q_rope, const float* w_in, float softmax_scale,
                float head_scale, uint8_t* q_codes, void* q_scales, float* w_out,
                const float* cos_sin, int32_t max_pos, int32_t dtype, int32_t* dev_status,
                cudaStream_t stream);

/*
 * Paged MQA logits ([P1] "Purpose", "Performance and accuracy"; [P2] "Purpose": the
 * scorer reads the cache in place, without gathering K first):
 *   logits[t * ld_logits + s] = sum_h w[t,h] * ReLU(q[t,h] . k[s])     (MXFP4)
 *   logits[t * ld_logits + s] = kscale[s] * sum_h w[t,h] * ReLU(q[t,h] . k[s])   (FP8)
 * for 0 <= s < visible(t); other entries of the row are not written.
 * Sequences: B of them; sequence b owns queries cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
 *   (int32 [B+1], cu_seqlens_q[0] = 0, cu_seqlens_q[B] = T) and seq_lens_k[b] keys
 *   (int32 [B]); key s of sequence b lives in page page_table[b*pt_stride + s/P], row s%P.
 *   causal = 0: visible(t) = seq_lens_k[b]; causal = 1: the n_q queries are the last n_q
 *   tokens of the sequence and query i sees keys 0 .. seq_lens_k[b] - n_q + i.
 * max_q_len: an upper bound of the queries per sequence (<= 1 selects the decode kernel);
 * max_seq_len_k: an upper bound of seq_lens_k (sizes the grid).
 * A sequence whose key count is negative or above max_seq_len_k, or whose query count
 * (cu_seqlens_q[b+1] - cu_seqlens_q[b]) is negative or above max_q_len, is skipped (none
 * of its logits are written) and sets IDX_STATUS_BAD_LEN.
 * q_codes / q_scales / w as produced by idx_q_quant (w = its w_out).
 * H: 1..64 for MXFP4 and FP8. ld_logits >= max visible, a multiple of 4 and at most
 * INT32_MAX / 32 (IDX_EUNSUPPORTED otherwise); logits fp32, 16-byte aligned.
 * Products are exact in the tensor core; sums are fp32. Accuracy against the exact
 * (fp64) scores: |error| <= 1e-4 * max_s |logit[t,s]| per row.
 * workspace (optional, may be NULL): at least idx_mqa_logits_workspace_bytes() bytes of device
 *   memory, 16-byte aligned, zero-filled by the caller before its first use; every call leaves
 *   it zero again. With it, a decode call (max_q_len <= 1) with at most 256 sequences hands the
 *   (sequence, 128-key tile) units out dynamically: each CTA claims small jobs from a counter
 *   there, so CTAs that start late take less work. The logits are the same either way. One
 *   workspace serves one call at a time (calls that overlap on the GPU need their own).
 */
int idx_mqa_logits_workspace_bytes(size_t* bytes);

int idx_mqa_logits_paged(const uint8_t* q_codes, const void* q_scales, const float* w,
                         int64_t T, int32_t H, int32_t dtype, const void* pool,
                         int64_t num_pages, int32_t page_size, int64_t page_stride,
                         const int32_t* page_table, int32_t pt_stride,
                         const int32_t* seq_lens_k, const int32_t* cu_seqlens_q, int32_t B,
                         int32_t causal, int32_t max_q_len, int32_t max_seq_len_k,
                         float* logits, int64_t ld_logits, void* workspace,
                         size_t workspace_bytes, int32_t* dev_status,
                         cudaStream_t stream);

/*
 * Per-query top-k ([P2] "Test Result / GPQA Diamond": the indexer picks top-k keys per
 * query once the context passes top-k x compress ratio; [P3] "Purpose":
 * topk_indices_buffer): out_idx[t*k .. t*k+k-1] = the logical key indices of the k largest
 * logits[t, 0 .. visible(t)-1] (same visible rule and arguments as the scorer). The set is
 * exact for the fp32 logits given; its order is: indices of values above the k-th value in
 * increasing index order, then indices equal to it in increasing index order. If
 * visible(t) < k all visible indices are returned, followed by -1 padding.
 * 1 <= k <= 4096; ld_logits <= INT32_MAX (IDX_EUNSUPPORTED otherwise). logits is a
 * 4-byte aligned device buffer and 0 <= max_seq_len_k <= ld_logits (IDX_EINVAL otherwise).
 * max_seq_len_k is the scorer's bound: a row whose sequence has a negative key count or one
 * above max_seq_len_k gets -1 in all k slots and sets IDX_STATUS_BAD_LEN in *dev_status
 * (when non-NULL), so no row is ever read past max_seq_len_k <= ld_logits. A row that
 * belongs to no sequence gets -1 in all k slots.
 */
int idx_topk(const float* logits, int64_t ld_logits, const int32_t* seq_lens_k,
             const int32_t* cu_seqlens_q, int32_t B, int64_t T, int32_t causal,
             int32_t max_seq_len_k, int32_t k, int32_t* out_idx, int32_t* dev_status,
             cudaStream_t stream);

/*
 * Candidate-pool scoring and top-k, the second level of DeepSeek-V4.1's two-level indexer
 * ([P2] "Purpose": the MXFP4 indexer's candidate-pool path, beside the dense path that scores
 * the whole context; [P2] "Scoring and metadata": the dense path is the scorer called with no
 * candidate blocks). A candidate block is one page-table block: block j of a sequence holds its
 * keys j*P .. j*P + P - 1. Query t lists n_cand[t] block ids at cand_blocks[t*cand_stride ..];
 * its candidate keys are its visible keys (as in idx_mqa_logits_paged) whose block is listed
 * (repeated ids count once; ids naming no visible block add nothing). out_idx[t*k .. t*k+k-1]
 * holds the key positions (in the sequence) of the k largest logits among the candidate keys,
 * -1 past their count; the logits are the ones idx_mqa_logits_paged computes. The choice of the
 * blocks (the first level) is the caller's.
 * Arguments as idx_mqa_topk_paged, plus: cand_blocks int32 [T][cand_stride], n_cand int32 [T],
 *   1 <= max_cand <= 1024 with max_cand <= cand_stride: an upper bound of n_cand[t]. A row whose
 *   n_cand is negative or above max_cand, or whose sequence breaks the length bounds, gets -1
 *   in all k slots and sets IDX_STATUS_BAD_LEN.
 * workspace: at least idx_mqa_topk_cand_workspace_bytes(T, max_cand, page_size, max_seq_len_k)
 *   bytes, 256-byte aligned; nothing in it needs a starting value. One workspace serves one
 *   call at a time. Four launches on the stream: candidate preparation, the decode scorer on
 *   one virtual sequence per query (the candidate blocks back to back), top-k, index mapping.
 */
int idx_mqa_topk_cand_workspace_bytes(int64_t T, int32_t max_cand, int32_t page_size,
                                      int32_t max_seq_len_k, size_t* bytes);

int idx_mqa_topk_cand_paged(const uint8_t* q_codes, const void* q_scales, const float* w,
                            int64_t T, int32_t H, int32_t dtype, const void* pool,
                            int64_t num_pages, int32_t page_size, int64_t page_stride,
                            const int32_t* page_table, int32_t pt_stride,
                            const int32_t* seq_lens_k, const int32_t* cu_seqlens_q, int32_t B,
                            int32_t causal, int32_t max_q_len, int32_t max_seq_len_k,
                            const int32_t* cand_blocks, int32_t cand_stride,
                            const int32_t* n_cand, int32_t max_cand, int32_t k, int32_t* out_idx,
                            void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            cudaStream_t stream);

/*
 * Paged MQA logits and per-query top-k in one launch ([P2] "Purpose": the cache is scored in
 * place; [P3] "Purpose": topk_indices_buffer). out_idx[t*k .. t*k+k-1] is what
 * idx_mqa_logits_paged followed by idx_topk (same arguments, k, max_seq_len_k) would give:
 * the same set in the same order, since both select on the same fp32 logits. The logits
 * matrix is never written to caller memory: decode (max_q_len <= 1) scores into a per-query
 * scratch row of the workspace, and the CTA that finishes a sequence's last tiles selects its
 * top-k; prefill keeps one block of scratch rows per SM, and the CTA that owns a block of
 * queries selects their top-k at the end of the block.
 * Arguments as idx_mqa_logits_paged, plus 1 <= k <= 4096 and out_idx: int32 [T][k].
 * workspace: device memory of at least the size idx_mqa_topk_workspace_bytes gives for the
 *   same T, H, B, max_q_len and max_seq_len_k, 256-byte aligned, zero-filled by the caller
 *   before its first use (decode keeps per-sequence arrival counters there, and every call
 *   that completes leaves them at zero again; zero it again after a call that reported
 *   IDX_STATUS_TIMEOUT). One workspace serves one call at a time.
 * Rows of no sequence, rows with no visible key and rows of sequences that break the length
 * bounds (IDX_STATUS_BAD_LEN) get -1 in all k slots.
 */
int idx_mqa_topk_workspace_bytes(int64_t T, int32_t H, int32_t B, int32_t max_q_len,
                                 int32_t max_seq_len_k, size_t* bytes);

int idx_mqa_topk_paged(const uint8_t* q_codes, const void* q_scales, const float* w,
                       int64_t T, int32_t H, int32_t dtype, const void* pool, int64_t num_pages,
                       int32_t page_size, int64_t page_stride, const int32_t* page_table,
                       int32_t pt_stride, const int32_t* seq_lens_k,
                       const int32_t* cu_seqlens_q, int32_t B, int32_t causal,
                       int32_t max_q_len, int32_t max_seq_len_k, int32_t k, int32_t* out_idx,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status,
                       cudaStream_t stream);

/*
 * Verification hook: applies the device element encoders used by the store and quant
 * kernels to n fp32 values. kind 0: e2m1 of v (code in the low nibble, sign in bit 3),
 * kind 1: e4m3 of v (saturating). in and out are device buffers.
 */
int idx_debug_encode(int32_t kind, const float* in, int64_t n, uint8_t* out,
                     cudaStream_t stream);

/*
 * idx_mqa_topk_paged without a workspace, for callers that cannot allocate device memory
 * (code that must not allocate once it runs, or that only holds pointers to its own inputs
 * and outputs). The web pages have no counterpart of this entry point; it serves deployment.
 * Decode only (max_q_len <= 1); otherwise arguments, results and status bits as
 * idx_mqa_topk_paged, whose decode kernel it launches.
 * Working memory: an 8 MiB array in device memory that the library owns (a per-sequence
 *   counter for up to 16384 sequences, then T rows of roundup(max_seq_len_k, 4) fp32
 *   scratch logits in the remaining 8 MiB - 64 KiB). Every GPU that loads the library holds
 *   the array until the process exits. Larger B or T x row length: IDX_EUNSUPPORTED, before
 *   anything is enqueued. The call allocates nothing.
 * Set-up: the first call on a device, with that device current, resolves the array's device
 *   address (cudaGetSymbolAddress) and keeps it; make that first call before any stream
 *   capture.
 * Every call clears the counters (an asynchronous memset on `stream`) and then reuses the
 *   same array: calls that can overlap on the GPU (other streams, other threads) race on it
 *   and must be ordered by the caller.
 */
int idx_mqa_topk_paged_noalloc(const uint8_t* q_codes, const void* q_scales, const float* w,
                               int64_t T, int32_t H, int32_t dtype, const void* pool,
                               int64_t num_pages, int32_t page_size, int64_t page_stride,
                               const int32_t* page_table, int32_t pt_stride,
                               const int32_t* seq_lens_k, const int32_t* cu_seqlens_q,
                               int32_t B, int32_t causal, int32_t max_q_len,
                               int32_t max_seq_len_k, int32_t k, int32_t* out_idx,
                               int32_t* dev_status, cudaStream_t stream);

/*
 * Measurement hook: the dense tensor-core rate of the scorers' MMA kinds. Launches one CTA
 * per SM, each issuing iters x 8 MMAs (M = 128, N = 256, K = 64 block-scaled MXFP4 for
 * IDX_MXFP4, K = 32 e4m3 for IDX_FP8) on zero operands into one tensor-memory accumulator.
 * *flops_per_cta (host, may be NULL) receives the flops one CTA performs; the caller times
 * the launch on `stream` and divides by the SM count times that. dev_status as elsewhere.
 */
int idx_debug_mma_rate(int32_t dtype, int32_t iters, int32_t* dev_status, double* flops_per_cta,
                       cudaStream_t stream);

/*
 * Test hook for the bounded waits: one CTA whose thread waits, with the wait helper every
 * kernel of the library uses, for an mbarrier phase that nothing completes, gives up after
 * limit_us microseconds (1 .. 1000000) of global time, sets IDX_STATUS_TIMEOUT in *dev_status
 * and returns; the context stays usable. *dev_status: a device int32 (required).
 */
int idx_debug_wait_timeout(int32_t limit_us, int32_t* dev_status, cudaStream_t stream);

/* Human-readable name of an idx_status value (static string). */
const char* idx_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* IDX_H */
