// api.cu -- the extern "C" entry points of idx.h: argument validation, then one launch on
// the caller's stream. Nothing here allocates, frees or synchronises.
#include <algorithm>
#include <cmath>

#include <nvtx3/nvToolsExt.h>

#include "../../include/idx.h"
#include "kernels.h"

namespace {

// One NVTX range per entry point call (visible in Nsight timelines; near free otherwise).
struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range&) = delete;
    Range& operator=(const Range&) = delete;
};

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline bool valid_dtype(int32_t d) { return d == IDX_MXFP4 || d == IDX_FP8; }
inline bool valid_rope(int32_t r) {
    return r == IDX_ROPE_NONE || r == IDX_ROPE_NEOX || r == IDX_ROPE_INTERLEAVED;
}
inline int64_t page_bytes(int32_t dtype, int32_t P) { return (dtype == IDX_MXFP4 ? 68 : 132) * (int64_t)P; }
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? IDX_OK : IDX_ECUDA; }
constexpr size_t kLogitsWorkspaceBytes = 256;  // the decode schedule's two counters, padded

// common pool checks: page size, stride, alignment
int check_pool(int32_t dtype, const void* pool, int64_t num_pages, int32_t page_size,
               int64_t page_stride) {
    if (!valid_dtype(dtype)) return IDX_EINVAL;
    if (page_size != 64 && page_size != 128) return IDX_EUNSUPPORTED;
    if (num_pages < 0) return IDX_EINVAL;
    if (num_pages > 0 && !pool) return IDX_EINVAL;
    if (!aligned(pool, 16)) return IDX_EINVAL;
    if (page_stride < page_bytes(dtype, page_size) || page_stride % 16 != 0) return IDX_EINVAL;
    return IDX_OK;
}

}  // namespace

extern "C" {

int idx_debug_mma_rate(int32_t dtype, int32_t iters, int32_t* dev_status, double* flops_per_cta,
                       cudaStream_t stream) {
    if (!valid_dtype(dtype) || iters < 1) return IDX_EINVAL;
    if (flops_per_cta) *flops_per_cta = (double)idx::mma_rate_flops_per_iter(dtype) * iters;
    return cuda_status(idx::launch_mma_rate(dtype, iters, dev_status, stream));
}

int idx_debug_wait_timeout(int32_t limit_us, int32_t* dev_status, cudaStream_t stream) {
    if (!dev_status || limit_us < 1 || limit_us > 1000000) return IDX_EINVAL;
    return cuda_status(idx::launch_wait_timeout(limit_us, dev_status, stream));
}

const char* idx_status_string(int status) {
    switch (status) {
        case IDX_OK: return "ok";
        case IDX_EINVAL: return "invalid argument";
        case IDX_EUNSUPPORTED: return "unsupported size or mode";
        case IDX_ECUDA: return "CUDA launch error";
        default: return "unknown status";
    }
}

int idx_cache_layout(int32_t dtype, int32_t page_size, idx_layout* out) {
    if (!out || !valid_dtype(dtype)) return IDX_EINVAL;
    if (page_size != 64 && page_size != 128) return IDX_EUNSUPPORTED;
    const int64_t per_code = dtype == IDX_MXFP4 ? 64 : 128;
    out->page_size = page_size;
    out->bytes_per_token = (int32_t)(per_code + 4);
    out->code_offset = 0;
    out->code_bytes = per_code * page_size;
    out->scale_offset = out->code_bytes;
    out->scale_bytes = 4LL * page_size;
    out->page_bytes = out->code_bytes + out->scale_bytes;
    return IDX_OK;
}

}  // extern "C"

namespace {

// Host-side checks and argument packing shared by idx_k_store and idx_qk_prep.
int k_store_args(const uint16_t* k, int64_t n_rows, int64_t k_row_stride, const int64_t* slot_mapping,
                 const int32_t* positions, const float* cos_sin, int32_t max_pos, int32_t rope,
                 int32_t apply_norm, const float* gamma, const float* beta, float eps, int32_t dtype,
                 void* pool, int64_t num_pages, int32_t page_size, int64_t page_stride,
                 int32_t* dev_status, idx::KStoreArgs& a) {
    if (n_rows < 0 || !valid_rope(rope)) return IDX_EINVAL;
    int st = check_pool(dtype, pool, num_pages, page_size, page_stride);
    if (st != IDX_OK) return st;
    a = idx::KStoreArgs{};
    a.dtype = dtype;
    if (n_rows == 0) return IDX_OK;
    if (!k || !slot_mapping || !aligned(k, 16) || k_row_stride < 128 || k_row_stride % 8 != 0)
        return IDX_EINVAL;
    if (rope != IDX_ROPE_NONE && (!positions || !cos_sin || !aligned(cos_sin, 16) || max_pos <= 0))
        return IDX_EINVAL;
    if (apply_norm && !(eps >= 0.0f && std::isfinite(eps))) return IDX_EINVAL;
    a.k = k; a.n_rows = n_rows; a.k_row_stride = k_row_stride; a.slot_mapping = slot_mapping;
    a.positions = positions; a.cos_sin = cos_sin; a.max_pos = max_pos; a.rope = rope;
    a.apply_norm = apply_norm != 0; a.gamma = gamma; a.beta = beta; a.eps = eps;
    a.pool = static_cast<uint8_t*>(pool); a.num_pages = num_pages; a.page_size = page_size;
    a.page_stride = page_stride; a.dev_status = dev_status;
    return IDX_OK;
}

// Host-side checks and argument packing shared by idx_q_quant and idx_qk_prep.
int q_quant_args(const uint16_t* q, int64_t T, int32_t H, const int32_t* positions, const float* cos_sin,
                 int32_t max_pos, int32_t rope, const float* w_in, float softmax_scale,
                 float head_scale, int32_t dtype, uint8_t* q_codes, void* q_scales, float* w_out,
                 int32_t* dev_status, idx::QQuantArgs& a) {
    if (T < 0 || !valid_rope(rope) || !valid_dtype(dtype)) return IDX_EINVAL;
    if (H < 1 || H > 64) return IDX_EUNSUPPORTED;
    a = idx::QQuantArgs{};
    a.dtype = dtype; a.H = H;
    if (T == 0) return IDX_OK;
    if (!q || !w_in || !q_codes || !w_out || !aligned(q, 16) || !aligned(q_codes, 16))
        return IDX_EINVAL;
    if (dtype == IDX_MXFP4 && (!q_scales || !aligned(q_scales, 16))) return IDX_EINVAL;
    if (q_scales && !aligned(q_scales, 4)) return IDX_EINVAL;
    if (rope != IDX_ROPE_NONE && (!positions || !cos_sin || !aligned(cos_sin, 16) || max_pos <= 0))
        return IDX_EINVAL;
    if (T > INT32_MAX) return IDX_EUNSUPPORTED;  // one grid column per token
    a.q = q; a.T = T; a.positions = positions; a.cos_sin = cos_sin;
    a.max_pos = max_pos; a.rope = rope; a.w_in = w_in;
    a.fold = (float)((double)softmax_scale * (double)head_scale);  // one rounding
    a.q_codes = q_codes; a.q_scales = q_scales; a.w_out = w_out; a.dev_status = dev_status;
    return IDX_OK;
}

}  // namespace

extern "C" {

int idx_k_store(const uint16_t* k, int64_t n_rows, int64_t k_row_stride,
                const int64_t* slot_mapping, const int32_t* positions, const float* cos_sin,
                int32_t max_pos, int32_t rope, int32_t apply_norm, const float* gamma,
                const float* beta, float eps, int32_t dtype, void* pool, int64_t num_pages,
                int32_t page_size, int64_t page_stride, int32_t* dev_status,
                cudaStream_t stream) {
    Range r("idx_k_store");
    idx::KStoreArgs a;
    const int st = k_store_args(k, n_rows, k_row_stride, slot_mapping, positions, cos_sin, max_pos, rope,
                                apply_norm, gamma, beta, eps, dtype, pool, num_pages, page_size,
                                page_stride, dev_status, a);
    if (st != IDX_OK || n_rows == 0) return st;
    return cuda_status(idx::launch_k_store(a, stream));
}

int idx_compress_k_store(const uint16_t* k_raw, const uint16_t* gate, int64_t n_raw, int64_t row_stride,
                         const int64_t* boundary, const int64_t* first, int64_t n_entries,
                         int32_t ratio, const int64_t* slot_mapping, const int32_t* positions,
                         const float* cos_sin, int32_t max_pos, int32_t rope, int32_t norm,
                         const float* gamma, const float* beta, float eps, int32_t dtype, void* pool,
                         int64_t num_pages, int32_t page_size, int64_t page_stride,
                         int32_t* dev_status, cudaStream_t stream) {
    Range r("idx_compress_k_store");
    if (n_raw < 0 || n_entries < 0 || !valid_rope(rope) || norm < 0 || norm > 2) return IDX_EINVAL;
    const int st = check_pool(dtype, pool, num_pages, page_size, page_stride);
    if (st != IDX_OK) return st;
    if (ratio < 1 || ratio > 128) return IDX_EUNSUPPORTED;
    if (n_entries == 0) return IDX_OK;
    if (!boundary || !first || !slot_mapping) return IDX_EINVAL;
    if (n_raw > 0 && (!k_raw || !gate || !aligned(k_raw, 16) || !aligned(gate, 16))) return IDX_EINVAL;
    if (row_stride < 128 || row_stride % 8 != 0) return IDX_EINVAL;
    if (rope != IDX_ROPE_NONE && (!positions || !cos_sin || !aligned(cos_sin, 16) || max_pos <= 0))
        return IDX_EINVAL;
    if (norm && !(eps >= 0.0f && std::isfinite(eps))) return IDX_EINVAL;
    idx::CompressArgs a{};
    a.k_raw = k_raw; a.gate = gate; a.n_raw = n_raw; a.row_stride = row_stride;
    a.boundary = boundary; a.first = first; a.n_entries = n_entries; a.ratio = ratio;
    a.slot_mapping = slot_mapping; a.positions = positions; a.cos_sin = cos_sin;
    a.max_pos = max_pos; a.rope = rope; a.norm = norm; a.dtype = dtype;
    a.gamma = gamma; a.beta = beta; a.eps = eps;
    a.pool = static_cast<uint8_t*>(pool); a.num_pages = num_pages; a.page_size = page_size;
    a.page_stride = page_stride; a.dev_status = dev_status;
    return cuda_status(idx::launch_compress(a, stream));
}

int idx_q_quant(const uint16_t* q, int64_t T, int32_t H, const int32_t* positions,
                const float* cos_sin, int32_t max_pos, int32_t rope, const float* w_in,
                float softmax_scale, float head_scale, int32_t dtype, uint8_t* q_codes,
                void* q_scales, float* w_out, int32_t* dev_status, cudaStream_t stream) {
    Range r("idx_q_quant");
    idx::QQuantArgs a;
    const int st = q_quant_args(q, T, H, positions, cos_sin, max_pos, rope, w_in, softmax_scale,
                                head_scale, dtype, q_codes, q_scales, w_out, dev_status, a);
    if (st != IDX_OK || T == 0) return st;
    return cuda_status(idx::launch_q_quant(a, stream));
}

int idx_qk_prep(const uint16_t* k, int64_t n_rows, int64_t k_row_stride, const int64_t* slot_mapping,
                const int32_t* k_positions, int32_t k_rope, int32_t apply_norm, const float* gamma,
                const float* beta, float eps, void* pool, int64_t num_pages, int32_t page_size,
                int64_t page_stride, const uint16_t* q, int64_t T, int32_t H,
                const int32_t* q_positions, int32_t q_rope, const float* w_in, float softmax_scale,
                float head_scale, uint8_t* q_codes, void* q_scales, float* w_out,
                const float* cos_sin, int32_t max_pos, int32_t dtype, int32_t* dev_status,
                cudaStream_t stream) {
    Range r("idx_qk_prep");
    idx::KStoreArgs ka;
    idx::QQuantArgs qa;
    int st = k_store_args(k, n_rows, k_row_stride, slot_mapping, k_positions, cos_sin, max_pos, k_rope,
                          apply_norm, gamma, beta, eps, dtype, pool, num_pages, page_size, page_stride,
                          dev_status, ka);
    if (st != IDX_OK) return st;
    st = q_quant_args(q, T, H, q_positions, cos_sin, max_pos, q_rope, w_in, softmax_scale, head_scale,
                      dtype, q_codes, q_scales, w_out, dev_status, qa);
    if (st != IDX_OK) return st;
    if (n_rows == 0 && T == 0) return IDX_OK;
    return cuda_status(idx::launch_qk_prep(ka, qa, stream));
}

int idx_mqa_logits_paged(const uint8_t* q_codes, const void* q_scales, const float* w,
                         int64_t T, int32_t H, int32_t dtype, const void* pool,
                         int64_t num_pages, int32_t page_size, int64_t page_stride,
                         const int32_t* page_table, int32_t pt_stride,
                         const int32_t* seq_lens_k, const int32_t* cu_seqlens_q, int32_t B,
                         int32_t causal, int32_t max_q_len, int32_t max_seq_len_k,
                         float* logits, int64_t ld_logits, void* workspace, size_t workspace_bytes,
                         int32_t* dev_status, cudaStream_t stream) {
    Range r("idx_mqa_logits_paged");
    int st = check_pool(dtype, pool, num_pages, page_size, page_stride);
    if (st != IDX_OK) return st;
    if (T < 0 || B < 0 || max_q_len < 0 || max_seq_len_k < 0 || pt_stride < 0) return IDX_EINVAL;
    if (H < 1 || H > 64) return IDX_EUNSUPPORTED;
    if (T == 0 || B == 0) return IDX_OK;
    if (!q_codes || !w || !page_table || !seq_lens_k || !cu_seqlens_q || !logits) return IDX_EINVAL;
    if (dtype == IDX_MXFP4 && (!q_scales || !aligned(q_scales, 16))) return IDX_EINVAL;
    if (!aligned(q_codes, 16) || !aligned(logits, 16) || ld_logits < max_seq_len_k ||
        ld_logits % 4 != 0)
        return IDX_EINVAL;
    if (pt_stride < (max_seq_len_k + page_size - 1) / page_size) return IDX_EINVAL;
    if (ld_logits > INT32_MAX / 32) return IDX_EUNSUPPORTED;  // 32-bit offsets inside a query block
    idx::ScoreArgs a{};
    a.q_codes = q_codes; a.q_scales = static_cast<const uint8_t*>(q_scales); a.w = w; a.T = T;
    a.H = H; a.dtype = dtype; a.pool = static_cast<const uint8_t*>(pool); a.num_pages = num_pages;
    a.page_size = page_size; a.page_stride = page_stride; a.page_table = page_table;
    a.pt_stride = pt_stride; a.seq_lens_k = seq_lens_k; a.cu_seqlens_q = cu_seqlens_q; a.B = B;
    a.causal = causal != 0; a.max_q_len = max_q_len; a.max_seq_len_k = max_seq_len_k;
    a.logits = logits; a.ld = ld_logits; a.dev_status = dev_status;
    if (workspace) {
        if (!aligned(workspace, 16) || workspace_bytes < kLogitsWorkspaceBytes) return IDX_EINVAL;
        a.counters = static_cast<int32_t*>(workspace);  // the dynamic decode schedule's counters
    }
    return cuda_status(idx::launch_scorer(a, stream));
}

int idx_mqa_logits_workspace_bytes(size_t* bytes) {
    if (!bytes) return IDX_EINVAL;
    *bytes = kLogitsWorkspaceBytes;
    return IDX_OK;
}

int idx_topk(const float* logits, int64_t ld_logits, const int32_t* seq_lens_k,
             const int32_t* cu_seqlens_q, int32_t B, int64_t T, int32_t causal,
             int32_t max_seq_len_k, int32_t k, int32_t* out_idx, int32_t* dev_status,
             cudaStream_t stream) {
    Range r("idx_topk");
    if (T < 0 || B < 0 || ld_logits < 0 || max_seq_len_k < 0) return IDX_EINVAL;
    if (k < 1 || k > 4096) return IDX_EUNSUPPORTED;
    if (T == 0) return IDX_OK;
    if (!logits || !seq_lens_k || !cu_seqlens_q || !out_idx || B == 0 || !aligned(logits, 4))
        return IDX_EINVAL;
    if (ld_logits > INT32_MAX) return IDX_EUNSUPPORTED;  // key indices are int32
    if (max_seq_len_k > ld_logits) return IDX_EINVAL;
    idx::TopkArgs a{};
    a.logits = logits; a.ld = ld_logits; a.seq_lens_k = seq_lens_k; a.cu_seqlens_q = cu_seqlens_q;
    a.B = B; a.T = T; a.causal = causal != 0; a.max_len = max_seq_len_k; a.k = k; a.out = out_idx;
    a.dev_status = dev_status;
    return cuda_status(idx::launch_topk(a, stream));
}

int idx_mqa_topk_workspace_bytes(int64_t T, int32_t H, int32_t B, int32_t max_q_len, int32_t max_seq_len_k,
                                 size_t* bytes) {
    if (!bytes || T < 0 || B < 0 || max_q_len < 0 || max_seq_len_k < 0) return IDX_EINVAL;
    if (H < 1 || H > 64) return IDX_EUNSUPPORTED;
    if (max_seq_len_k > INT32_MAX / 32) return IDX_EUNSUPPORTED;
    const int64_t n = idx::scorer_topk_workspace_bytes(T, H, B, max_q_len, max_seq_len_k);
    if (n < 0) return IDX_ECUDA;
    *bytes = (size_t)n;
    return IDX_OK;
}

int idx_mqa_topk_paged(const uint8_t* q_codes, const void* q_scales, const float* w, int64_t T, int32_t H,
                       int32_t dtype, const void* pool, int64_t num_pages, int32_t page_size,
                       int64_t page_stride, const int32_t* page_table, int32_t pt_stride,
                       const int32_t* seq_lens_k, const int32_t* cu_seqlens_q, int32_t B, int32_t causal,
                       int32_t max_q_len, int32_t max_seq_len_k, int32_t k, int32_t* out_idx,
                       void* workspace, size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream) {
    Range r("idx_mqa_topk_paged");
    int st = check_pool(dtype, pool, num_pages, page_size, page_stride);
    if (st != IDX_OK) return st;
    if (T < 0 || B < 0 || max_q_len < 0 || max_seq_len_k < 0 || pt_stride < 0) return IDX_EINVAL;
    if (H < 1 || H > 64 || k < 1 || k > 4096) return IDX_EUNSUPPORTED;
    if (max_seq_len_k > INT32_MAX / 32) return IDX_EUNSUPPORTED;
    if (T == 0) return IDX_OK;
    if (!out_idx || !seq_lens_k || !cu_seqlens_q || B == 0) return IDX_EINVAL;
    if (max_seq_len_k > 0 && (!q_codes || !w || !page_table)) return IDX_EINVAL;
    if (dtype == IDX_MXFP4 && max_seq_len_k > 0 && (!q_scales || !aligned(q_scales, 16))) return IDX_EINVAL;
    if ((q_codes && !aligned(q_codes, 16)) || !aligned(workspace, 256)) return IDX_EINVAL;
    if (pt_stride < (max_seq_len_k + page_size - 1) / page_size) return IDX_EINVAL;
    const int64_t need = idx::scorer_topk_workspace_bytes(T, H, B, max_q_len, max_seq_len_k);
    if (need < 0) return IDX_ECUDA;
    if (!workspace || (int64_t)workspace_bytes < need) return IDX_EINVAL;
    idx::ScoreArgs a{};
    a.q_codes = q_codes; a.q_scales = static_cast<const uint8_t*>(q_scales); a.w = w; a.T = T;
    a.H = H; a.dtype = dtype; a.pool = static_cast<const uint8_t*>(pool); a.num_pages = num_pages;
    a.page_size = page_size; a.page_stride = page_stride; a.page_table = page_table;
    a.pt_stride = pt_stride; a.seq_lens_k = seq_lens_k; a.cu_seqlens_q = cu_seqlens_q; a.B = B;
    a.causal = causal != 0; a.max_q_len = max_q_len; a.max_seq_len_k = max_seq_len_k;
    a.topk_k = k; a.out_idx = out_idx; a.dev_status = dev_status;
    return cuda_status(idx::launch_scorer_topk(a, workspace, stream));
}

int idx_debug_encode(int32_t kind, const float* in, int64_t n, uint8_t* out, cudaStream_t stream) {
    if ((kind != 0 && kind != 1) || n < 0) return IDX_EINVAL;
    if (n == 0) return IDX_OK;
    if (!in || !out) return IDX_EINVAL;
    return cuda_status(idx::launch_debug_encode(kind, in, n, out, stream));
}

}  // extern "C"

namespace {

// Workspace of the candidate path: cu' [T+1], vlen [T], the virtual page table and the sorted
// block ids [T][max_cand] (int32, each 256-byte padded), then the logits [T][ld'] with
// ld' = the longest virtual row (min(max_cand * P, max_seq_len_k)) rounded up to 4.
struct CandLayout {
    int64_t o_vlen, o_vpt, o_vblk, o_logits, total, ld, max_len;
};

CandLayout cand_layout(int64_t T, int32_t max_cand, int32_t page_size, int32_t max_seq_len_k) {
    auto up = [](int64_t x) { return (x + 255) / 256 * 256; };
    CandLayout l{};
    l.max_len = std::min<int64_t>((int64_t)max_cand * page_size, max_seq_len_k);
    l.ld = (std::max<int64_t>(l.max_len, 1) + 3) / 4 * 4;
    l.o_vlen = up(4 * (T + 1));
    l.o_vpt = l.o_vlen + up(4 * T);
    l.o_vblk = l.o_vpt + up(4 * T * max_cand);
    l.o_logits = l.o_vblk + up(4 * T * max_cand);
    l.total = l.o_logits + up(4 * T * l.ld);
    return l;
}

}  // namespace

extern "C" {

int idx_mqa_topk_cand_workspace_bytes(int64_t T, int32_t max_cand, int32_t page_size, int32_t max_seq_len_k,
                                      size_t* bytes) {
    if (!bytes || T < 0 || max_seq_len_k < 0) return IDX_EINVAL;
    if (page_size != 64 && page_size != 128) return IDX_EUNSUPPORTED;
    if (max_cand < 1 || max_cand > 1024 || max_seq_len_k > INT32_MAX / 32) return IDX_EUNSUPPORTED;
    *bytes = (size_t)cand_layout(T, max_cand, page_size, max_seq_len_k).total;
    return IDX_OK;
}

int idx_mqa_topk_cand_paged(const uint8_t* q_codes, const void* q_scales, const float* w, int64_t T, int32_t H,
                            int32_t dtype, const void* pool, int64_t num_pages, int32_t page_size,
                            int64_t page_stride, const int32_t* page_table, int32_t pt_stride,
                            const int32_t* seq_lens_k, const int32_t* cu_seqlens_q, int32_t B, int32_t causal,
                            int32_t max_q_len, int32_t max_seq_len_k, const int32_t* cand_blocks,
                            int32_t cand_stride, const int32_t* n_cand, int32_t max_cand, int32_t k,
                            int32_t* out_idx, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            cudaStream_t stream) {
    Range r("idx_mqa_topk_cand_paged");
    int st = check_pool(dtype, pool, num_pages, page_size, page_stride);
    if (st != IDX_OK) return st;
    if (T < 0 || B < 0 || max_q_len < 0 || max_seq_len_k < 0 || pt_stride < 0) return IDX_EINVAL;
    if (H < 1 || H > 64 || k < 1 || k > 4096) return IDX_EUNSUPPORTED;
    if (max_cand < 1 || max_cand > 1024 || max_seq_len_k > INT32_MAX / 32) return IDX_EUNSUPPORTED;
    if (cand_stride < max_cand) return IDX_EINVAL;
    if (T == 0) return IDX_OK;
    if (T > INT32_MAX - 1) return IDX_EUNSUPPORTED;  // one virtual sequence per query
    if (!out_idx || !seq_lens_k || !cu_seqlens_q || !cand_blocks || !n_cand || B == 0) return IDX_EINVAL;
    if (max_seq_len_k > 0 && (!q_codes || !w || !page_table)) return IDX_EINVAL;
    if (dtype == IDX_MXFP4 && max_seq_len_k > 0 && (!q_scales || !aligned(q_scales, 16))) return IDX_EINVAL;
    if ((q_codes && !aligned(q_codes, 16)) || !aligned(workspace, 256)) return IDX_EINVAL;
    if (pt_stride < (max_seq_len_k + page_size - 1) / page_size) return IDX_EINVAL;
    const CandLayout l = cand_layout(T, max_cand, page_size, max_seq_len_k);
    if (!workspace || (int64_t)workspace_bytes < l.total) return IDX_EINVAL;
    uint8_t* ws = static_cast<uint8_t*>(workspace);

    idx::CandArgs c{};
    c.cu_seqlens_q = cu_seqlens_q; c.seq_lens_k = seq_lens_k; c.page_table = page_table;
    c.pt_stride = pt_stride; c.B = B; c.causal = causal != 0; c.max_q_len = max_q_len;
    c.max_seq_len_k = max_seq_len_k; c.page_size = page_size; c.T = T; c.cand = cand_blocks;
    c.cand_stride = cand_stride; c.max_cand = max_cand; c.n_cand = n_cand;
    c.vcu = reinterpret_cast<int32_t*>(ws);
    c.vlen = reinterpret_cast<int32_t*>(ws + l.o_vlen);
    c.vpt = reinterpret_cast<int32_t*>(ws + l.o_vpt);
    c.vblk = reinterpret_cast<int32_t*>(ws + l.o_vblk);
    c.dev_status = dev_status;
    cudaError_t e = idx::launch_cand_prep(c, stream);
    if (e != cudaSuccess) return IDX_ECUDA;

    // the decode scorer over one virtual sequence per query; its prologue reads the virtual
    // lengths and page table, so it starts after the preparation has finished
    idx::ScoreArgs a{};
    a.q_codes = q_codes; a.q_scales = static_cast<const uint8_t*>(q_scales); a.w = w; a.T = T;
    a.H = H; a.dtype = dtype; a.pool = static_cast<const uint8_t*>(pool); a.num_pages = num_pages;
    a.page_size = page_size; a.page_stride = page_stride; a.page_table = c.vpt; a.pt_stride = max_cand;
    a.seq_lens_k = c.vlen; a.cu_seqlens_q = c.vcu; a.B = (int32_t)T; a.causal = 0; a.max_q_len = 1;
    a.max_seq_len_k = (int32_t)l.max_len; a.logits = reinterpret_cast<float*>(ws + l.o_logits); a.ld = l.ld;
    a.dev_status = dev_status; a.no_pdl = true;
    e = idx::launch_scorer_decode(a, stream);
    if (e != cudaSuccess) return IDX_ECUDA;

    idx::TopkArgs tk{};
    tk.logits = a.logits; tk.ld = l.ld; tk.seq_lens_k = c.vlen; tk.cu_seqlens_q = c.vcu; tk.B = (int32_t)T;
    tk.T = T; tk.causal = 0; tk.max_len = (int32_t)l.max_len; tk.k = k; tk.out = out_idx; tk.dev_status = dev_status;
    e = idx::launch_topk(tk, stream);
    if (e != cudaSuccess) return IDX_ECUDA;
    return cuda_status(idx::launch_cand_map(c.vblk, max_cand, page_size, T, k, out_idx, stream));
}

}  // extern "C"

namespace idx {
// Scorer dispatch: one kernel family per dtype.
cudaError_t launch_scorer(const ScoreArgs& a, cudaStream_t st) {
    if (a.max_q_len <= 1) return launch_scorer_decode(a, st);
    return launch_scorer_prefill(a, st);
}

namespace {
int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
int64_t scratch_ld(int32_t max_seq_len_k) { return round_up(max_seq_len_k > 0 ? max_seq_len_k : 1, 4); }
}  // namespace

// Workspace of the fused scorer -> top-k. Decode (max_q_len <= 1): per-sequence arrival
// counters [B] int32 (256-byte padded), then a logits scratch row per query [T][ld]. Prefill:
// one block of scratch rows per CTA [SMs][QB][ld], QB = queries per block for H heads.
int64_t scorer_topk_workspace_bytes(int64_t T, int32_t H, int32_t B, int32_t max_q_len, int32_t max_seq_len_k) {
    const int64_t ld = scratch_ld(max_seq_len_k);
    if (max_q_len <= 1) return round_up(4 * (int64_t)B, 256) + 4 * T * ld;
    const int sms = device_sm_count();
    if (sms <= 0) return -1;
    return 4 * (int64_t)sms * prefill_queries_per_block(H) * ld;
}

cudaError_t launch_scorer_topk(const ScoreArgs& a0, void* workspace, cudaStream_t st) {
    ScoreArgs a = a0;
    a.ld = scratch_ld(a.max_seq_len_k);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (a.max_q_len <= 1) {
        a.counters = reinterpret_cast<int32_t*>(ws);
        a.logits = reinterpret_cast<float*>(ws + round_up(4 * (int64_t)a.B, 256));
        return launch_scorer_decode_select(a, st);
    }
    a.counters = nullptr;
    a.logits = reinterpret_cast<float*>(ws);
    return launch_scorer_prefill_select(a, st);
}
}  // namespace idx
