// cand.cu -- the candidate-pool path of the indexer (the second level of DeepSeek-V4.1's
// two-level indexer): each query scores and ranks only the keys of its candidate blocks.
//
// vllm PR 60834 "Purpose": besides the dense path, which scores the whole context, the MXFP4
// indexer has a candidate-pool path that exists for V4.1's two-level indexer; the dense path
// is the scorer called with no candidate blocks ("Scoring and metadata"). A candidate block is
// one page-table block of P keys; the first level that picks the blocks is the caller's.
//
// The path reuses the paged scorer and the top-k unchanged, through a virtual page table:
//   cand_prep_kernel  one warp per query: its block ids, those naming no visible block
//                     dropped, deduplicated and sorted (ids in shared memory; a kept id's
//                     slot is the count of kept ids below it); the virtual page table row
//                     (the sorted blocks' physical pages), the sorted ids, the virtual length
//                     and cu' = 0, 1, .., T;
//   decode scorer     one virtual sequence per query (its candidate keys back to back; only
//                     the last block can be partial, since it holds the visibility edge);
//   top-k             over the virtual rows;
//   cand_map_kernel   virtual position v -> key position blk[v / P] * P + v % P.
// The scorer's prologue reads lengths and the page table before its grid-dependency wait, so
// here it is launched as an ordinary stream-ordered launch after cand_prep_kernel. The top-k,
// whose prologue reads the virtual lengths too, starts no earlier than the scorer, so
// cand_prep_kernel has completed by then.
#include "common.cuh"
#include "kernels.h"

namespace idx {

namespace {

constexpr int kPrepWarps = 4;

__global__ void __launch_bounds__(32 * kPrepWarps) cand_prep_kernel(CandArgs a) {
    extern __shared__ int32_t s_ids[];  // [kPrepWarps][max_cand]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * kPrepWarps + warp;
    if (t >= a.T) return;
    int32_t* ids = s_ids + warp * a.max_cand;
    int32_t* vpt = a.vpt + t * a.max_cand;
    int32_t* vblk = a.vblk + t * a.max_cand;
    if (lane == 0) {
        a.vcu[t] = (int32_t)t;
        if (t == a.T - 1) a.vcu[a.T] = (int32_t)a.T;
    }
    // the query's sequence and visible keys (rows of no sequence, or of one whose lengths
    // break their bounds, keep no candidate)
    const int b = seq_of_query(a.cu_seqlens_q, a.B, t);
    int64_t vis = 0;
    bool ok = b >= 0;
    int32_t n = ok ? a.n_cand[t] : 0;
    if (ok) {
        const int64_t q0 = a.cu_seqlens_q[b], nq = a.cu_seqlens_q[b + 1] - q0;
        const int32_t len = a.seq_lens_k[b];
        if (len < 0 || len > a.max_seq_len_k || nq > a.max_q_len || n < 0 || n > a.max_cand) {
            if (lane == 0) report(a.dev_status, IDX_STATUS_BAD_LEN);
            ok = false;
        } else {
            vis = visible_keys(len, nq, t - q0, a.causal);
        }
    }
    if (!ok) n = 0;
    const int32_t nblk = (int32_t)((vis + a.page_size - 1) / a.page_size);
    const int32_t* c = a.cand + t * a.cand_stride;
    for (int i = lane; i < n; i += 32) {
        const int32_t id = c[i];
        ids[i] = (id >= 0 && id < nblk) ? id : -1;  // -1: names no visible block
    }
    __syncwarp();
    // repeats are dropped: an id is kept at its first occurrence (chunks of 32, every lane
    // decides before any lane writes)
    for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + lane;
        bool dup = false;
        if (i < n) {
            const int32_t id = ids[i];
            if (id >= 0)
                for (int j = 0; j < i && !dup; ++j) dup = ids[j] == id;
        }
        __syncwarp();
        if (dup) ids[i] = -1;
        __syncwarp();
    }
    // a kept id's slot is the number of kept ids below it
    int32_t kept = 0, top = -1;
    for (int i = lane; i < n; i += 32) {
        const int32_t id = ids[i];
        if (id < 0) continue;
        int32_t rank = 0;
        for (int j = 0; j < n; ++j) {
            const int32_t o = ids[j];
            rank += (o >= 0) & (o < id);
        }
        vblk[rank] = id;
        vpt[rank] = a.page_table[(int64_t)b * a.pt_stride + id];
        ++kept;
        top = max(top, id);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        kept += __shfl_xor_sync(kFull, kept, off);
        top = max(top, __shfl_xor_sync(kFull, top, off));
    }
    if (lane == 0) {
        // every kept block but the highest lies wholly below the visibility edge
        const int64_t last = vis - (int64_t)top * a.page_size;
        a.vlen[t] = kept == 0 ? 0 : (int32_t)((int64_t)(kept - 1) * a.page_size + (last < a.page_size ? last : a.page_size));
    }
}

__global__ void cand_map_kernel(const int32_t* vblk, int32_t max_cand, int32_t page_size, int64_t T,
                                int32_t k, int32_t* out) {
    const int64_t n = T * k;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = out[i];
        if (v < 0) continue;
        const int64_t t = i / k;
        out[i] = vblk[t * max_cand + v / page_size] * page_size + v % page_size;
    }
}

}  // namespace

cudaError_t launch_cand_prep(const CandArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    const int64_t grid = (a.T + kPrepWarps - 1) / kPrepWarps;
    const size_t smem = (size_t)kPrepWarps * a.max_cand * sizeof(int32_t);
    cudaError_t e = cudaFuncSetAttribute(cand_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(false, cand_prep_kernel, dim3((unsigned)grid), dim3(32 * kPrepWarps), smem, st, a);
}

cudaError_t launch_cand_map(const int32_t* vblk, int32_t max_cand, int32_t page_size, int64_t T, int32_t k,
                            int32_t* out_idx, cudaStream_t st) {
    const int64_t n = T * k;
    if (n == 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    return launch_k(false, cand_map_kernel, dim3((unsigned)blocks), dim3(256), 0, st, vblk, max_cand, page_size,
                    T, k, out_idx);
}

}  // namespace idx
