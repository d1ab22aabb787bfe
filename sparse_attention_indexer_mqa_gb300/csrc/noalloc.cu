// noalloc.cu -- idx_mqa_topk_paged_noalloc: the decode form of the fused scorer -> top-k
// (idx_mqa_topk_paged) with its working memory in a fixed device array that belongs to this
// library, for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs where allocation
// is not allowed (inside a region whose memory plan is fixed up front, under an allocator
// that forbids new device allocations after start-up), or a host that only holds pointers to
// its own inputs and outputs. For them the arrival counters and the logits scratch rows live
// in g_noalloc_scratch below, a static array of kNoAllocBytes in device memory: every GPU
// that loads the library holds it until the process exits. The entry point itself calls no
// cudaMalloc, cudaFree or allocating routine.
//
// In host code the name g_noalloc_scratch is only a host-side stand-in for the array, not a
// device address: handing it to a kernel would fault, or on a GPU that can reach host memory
// silently use the wrong memory. So the first call on each device, with that device current,
// asks the runtime for the array's device address (cudaGetSymbolAddress) and keeps it; later
// calls on that device reuse it, and the kernels receive that address as an argument.
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/idx.h"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocBytes = size_t(8) << 20;   // 8 MiB
constexpr int kNoAllocMaxSeqs = 16384;              // arrival counters, one per sequence
constexpr size_t kCounterBytes = 4 * (size_t)kNoAllocMaxSeqs;  // 64 KiB, 256-byte aligned

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device

// The array's device address on the current device (resolved once per device).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" int idx_mqa_topk_paged_noalloc(const uint8_t* q_codes, const void* q_scales, const float* w,
                                          int64_t T, int32_t H, int32_t dtype, const void* pool,
                                          int64_t num_pages, int32_t page_size, int64_t page_stride,
                                          const int32_t* page_table, int32_t pt_stride,
                                          const int32_t* seq_lens_k, const int32_t* cu_seqlens_q, int32_t B,
                                          int32_t causal, int32_t max_q_len, int32_t max_seq_len_k, int32_t k,
                                          int32_t* out_idx, int32_t* dev_status, cudaStream_t stream) {
    nvtxRangePushA("idx_mqa_topk_paged_noalloc");
    struct Pop {
        ~Pop() { nvtxRangePop(); }
    } pop;
    // the same argument rules as idx_mqa_topk_paged
    if (dtype != IDX_MXFP4 && dtype != IDX_FP8) return IDX_EINVAL;
    if (page_size != 64 && page_size != 128) return IDX_EUNSUPPORTED;
    if (num_pages < 0 || (num_pages > 0 && !pool) || !aligned16(pool)) return IDX_EINVAL;
    if (page_stride < (dtype == IDX_MXFP4 ? 68 : 132) * (int64_t)page_size || page_stride % 16 != 0)
        return IDX_EINVAL;
    if (T < 0 || B < 0 || max_q_len < 0 || max_seq_len_k < 0 || pt_stride < 0) return IDX_EINVAL;
    if (H < 1 || H > 64 || k < 1 || k > 4096) return IDX_EUNSUPPORTED;
    if (max_seq_len_k > INT32_MAX / 32) return IDX_EUNSUPPORTED;
    // decode only (one query per sequence), and the scratch must fit the fixed array
    if (max_q_len > 1 || B > kNoAllocMaxSeqs) return IDX_EUNSUPPORTED;
    const int64_t ld = ((max_seq_len_k > 0 ? max_seq_len_k : 1) + 3) / 4 * 4;
    if (T > (int64_t)((kNoAllocBytes - kCounterBytes) / 4) / ld) return IDX_EUNSUPPORTED;
    if (T == 0) return IDX_OK;
    if (!out_idx || !seq_lens_k || !cu_seqlens_q || B == 0) return IDX_EINVAL;
    if (max_seq_len_k > 0 && (!q_codes || !w || !page_table)) return IDX_EINVAL;
    if (dtype == IDX_MXFP4 && max_seq_len_k > 0 && (!q_scales || !aligned16(q_scales))) return IDX_EINVAL;
    if (q_codes && !aligned16(q_codes)) return IDX_EINVAL;
    if (pt_stride < (max_seq_len_k + page_size - 1) / page_size) return IDX_EINVAL;

    void* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return IDX_ECUDA;
    // the counters must start at zero: the array keeps whatever the previous call left
    if (cudaMemsetAsync(base, 0, 4 * (size_t)B, stream) != cudaSuccess) return IDX_ECUDA;
    idx::ScoreArgs a{};
    a.q_codes = q_codes; a.q_scales = static_cast<const uint8_t*>(q_scales); a.w = w; a.T = T;
    a.H = H; a.dtype = dtype; a.pool = static_cast<const uint8_t*>(pool); a.num_pages = num_pages;
    a.page_size = page_size; a.page_stride = page_stride; a.page_table = page_table;
    a.pt_stride = pt_stride; a.seq_lens_k = seq_lens_k; a.cu_seqlens_q = cu_seqlens_q; a.B = B;
    a.causal = causal != 0; a.max_q_len = max_q_len; a.max_seq_len_k = max_seq_len_k;
    a.topk_k = k; a.out_idx = out_idx; a.dev_status = dev_status;
    a.counters = static_cast<int32_t*>(base);
    a.logits = reinterpret_cast<float*>(static_cast<uint8_t*>(base) + kCounterBytes);
    a.ld = ld;
    return idx::launch_scorer_decode_select(a, stream) == cudaSuccess ? IDX_OK : IDX_ECUDA;
}
