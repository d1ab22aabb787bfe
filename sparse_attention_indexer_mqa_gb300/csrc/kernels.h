// kernels.h -- internal argument blocks and launchers behind the C ABI (idx.h).
// The ABI layer validates every argument before it fills one of these.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace idx {

struct KStoreArgs {
    const uint16_t* k;
    int64_t n_rows, k_row_stride;
    const int64_t* slot_mapping;
    const int32_t* positions;
    const float* cos_sin;
    int32_t max_pos, rope, apply_norm, dtype;
    const float* gamma;
    const float* beta;
    float eps;
    uint8_t* pool;
    int64_t num_pages;
    int32_t page_size;
    int64_t page_stride;
    int32_t* dev_status;
};

// Compressed K store: entries pool raw rows (see idx_compress_k_store).
struct CompressArgs {
    const uint16_t* k_raw;
    const uint16_t* gate;
    int64_t n_raw, row_stride;
    const int64_t* boundary;
    const int64_t* first;
    int64_t n_entries;
    int32_t ratio;
    const int64_t* slot_mapping;
    const int32_t* positions;
    const float* cos_sin;
    int32_t max_pos, rope, norm, dtype;
    const float* gamma;
    const float* beta;
    float eps;
    uint8_t* pool;
    int64_t num_pages;
    int32_t page_size;
    int64_t page_stride;
    int32_t* dev_status;
};

struct QQuantArgs {
    const uint16_t* q;
    int64_t T;  // tokens; each has H heads (Hq = H rounded up to 8 in the image)
    int32_t H;
    const int32_t* positions;
    const float* cos_sin;
    int32_t max_pos, rope, dtype;
    const float* w_in;
    float fold;  // fp32(softmax_scale * head_scale)
    uint8_t* q_codes;
    void* q_scales;
    float* w_out;
    int32_t* dev_status;
};

struct ScoreArgs {
    const uint8_t* q_codes;
    const uint8_t* q_scales;  // MXFP4: E8M0 scale atoms [T][512]; FP8: unused
    const float* w;           // [T][H]
    int64_t T;
    int32_t H, dtype;
    const uint8_t* pool;
    int64_t num_pages;
    int32_t page_size;
    int64_t page_stride;
    const int32_t* page_table;
    int32_t pt_stride;
    const int32_t* seq_lens_k;
    const int32_t* cu_seqlens_q;
    int32_t B, causal, max_q_len, max_seq_len_k;
    float* logits;  // select mode: the workspace's logits scratch (see launch_scorer_topk)
    int64_t ld;
    int32_t* dev_status;
    // select mode only (idx_mqa_topk_paged): top-k size, output [T][topk_k], per-sequence
    // arrival counters of the decode kernel (zero before and after a call)
    int32_t topk_k;
    int32_t* out_idx;
    int32_t* counters;
    // launch without programmatic dependent launch: set when the previous kernel on the
    // stream writes this call's metadata (lengths, page table), which the scorer's prologue
    // reads before its grid-dependency wait
    bool no_pdl;
};

struct TopkArgs {
    const float* logits;
    int64_t ld;
    const int32_t* seq_lens_k;
    const int32_t* cu_seqlens_q;
    int32_t B;
    int64_t T;
    int32_t causal, max_len, k;  // max_len: the scorer's max_seq_len_k (<= ld)
    int32_t* out;
    int32_t* dev_status;
};

cudaError_t launch_k_store(const KStoreArgs& a, cudaStream_t st);
cudaError_t launch_q_quant(const QQuantArgs& a, cudaStream_t st);
cudaError_t launch_qk_prep(const KStoreArgs& ka, const QQuantArgs& qa, cudaStream_t st);
cudaError_t launch_compress(const CompressArgs& a, cudaStream_t st);

// Candidate-pool scoring (idx_mqa_topk_cand_paged): per query, its candidate blocks sorted and
// deduplicated into a virtual page table; the decode scorer and top-k then run on one virtual
// sequence per query, and the indices are mapped back to key positions.
struct CandArgs {
    const int32_t* cu_seqlens_q;
    const int32_t* seq_lens_k;
    const int32_t* page_table;
    int32_t pt_stride, B, causal, max_q_len, max_seq_len_k, page_size;
    int64_t T;
    const int32_t* cand;
    int32_t cand_stride, max_cand;
    const int32_t* n_cand;
    // workspace: cu' [T+1], vlen [T], virtual page table and sorted blocks [T][max_cand]
    int32_t* vcu;
    int32_t* vlen;
    int32_t* vpt;
    int32_t* vblk;
    int32_t* dev_status;
};
cudaError_t launch_cand_prep(const CandArgs& a, cudaStream_t st);
cudaError_t launch_cand_map(const int32_t* vblk, int32_t max_cand, int32_t page_size, int64_t T, int32_t k,
                            int32_t* out_idx, cudaStream_t st);
cudaError_t launch_debug_encode(int kind, const float* in, int64_t n, uint8_t* out, cudaStream_t st);
cudaError_t launch_scorer(const ScoreArgs& a, cudaStream_t st);
cudaError_t launch_scorer_decode(const ScoreArgs& a, cudaStream_t st);
cudaError_t launch_scorer_prefill(const ScoreArgs& a, cudaStream_t st);
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st);

// Fused scorer -> top-k (idx_mqa_topk_paged): bytes of workspace it needs, and the launch.
int64_t scorer_topk_workspace_bytes(int64_t T, int32_t H, int32_t B, int32_t max_q_len, int32_t max_seq_len_k);
cudaError_t launch_scorer_topk(const ScoreArgs& a, void* workspace, cudaStream_t st);
cudaError_t launch_scorer_decode_select(const ScoreArgs& a, cudaStream_t st);
cudaError_t launch_scorer_prefill_select(const ScoreArgs& a, cudaStream_t st);
int prefill_queries_per_block(int32_t H);
int device_sm_count();

// Bounded-wait test hook (idx_debug_wait_timeout).
cudaError_t launch_wait_timeout(int32_t limit_us, int32_t* status, cudaStream_t st);

// Dense tensor-core rate probe (idx_debug_mma_rate): one CTA per SM, `iters` loop iterations.
cudaError_t launch_mma_rate(int32_t dtype, int32_t iters, int32_t* status, cudaStream_t st);
int mma_rate_flops_per_iter(int32_t dtype);

}  // namespace idx
