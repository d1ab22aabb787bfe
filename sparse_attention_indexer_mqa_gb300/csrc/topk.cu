// topk.cu -- per-query top-k over the indexer logits by radix select.
//
// vllm PR 60834 "Test Result / GPQA Diamond": the indexer keeps the top-k (1024) keys per
// query once the context exceeds top-k x compress ratio; vllm PR 53094 "Purpose" names the
// per-token topk_indices_buffer it fills. The set of the k largest logits is unique up to
// ties at the k-th value; this kernel returns the indices above the k-th value, then the
// indices equal to it, each group in increasing index order, so the result is
// deterministic.
//
// One CTA (1024 threads) per query row. The row's logits are read from global memory once,
// mapped to order-preserving uint32 keys and kept in shared memory (rows longer than the
// shared-memory capacity are re-read from global memory instead). Three histogram passes
// (11, 11, 10 bits, shared-memory atomics) fix the k-th key exactly; the final pass gives
// each thread a contiguous chunk of the row, so one block-wide scan orders the output.
#include "common.cuh"
#include "kernels.h"

namespace idx {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int64_t kSmemKeysMax = 48 * 1024;  // 192 KB of keys

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive sum scan over the CTA; `total` receives the CTA-wide sum.
template <typename T>
__device__ __forceinline__ T block_scan(T v, T* warp_sums, T& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
        T s = lane < kWarps ? warp_sums[lane] : T(0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            T y = __shfl_up_sync(kFull, s, o);
            if (lane >= o) s += y;
        }
        if (lane < kWarps) warp_sums[lane] = s;
    }
    __syncthreads();
    const T add = w > 0 ? warp_sums[w - 1] : T(0);
    total = warp_sums[kWarps - 1];
    __syncthreads();
    return x + add;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a, int64_t smem_keys) {
    extern __shared__ uint32_t skeys[];
    __shared__ uint32_t hist[2048];
    __shared__ uint64_t warp_sums[kWarps];
    __shared__ uint32_t sel_bin, sel_above;

    const int64_t t = blockIdx.x;
    const int b = seq_of_query(a.cu_seqlens_q, a.B, t);
    int64_t vis = 0;
    if (b >= 0) {
        const int64_t q0 = a.cu_seqlens_q[b], nq = a.cu_seqlens_q[b + 1] - q0;
        vis = visible_keys(a.seq_lens_k[b], nq, t - q0, a.causal);
    }
    int32_t* out = a.out + t * a.k;
    const float* row = a.logits + t * a.ld;
    if (vis <= a.k) {
        for (int i = threadIdx.x; i < a.k; i += kThreads) out[i] = i < vis ? i : -1;
        return;
    }
    const bool cached = vis <= smem_keys;
    auto key_at = [&](int64_t i) -> uint32_t { return cached ? skeys[i] : order_key(row[i]); };

    uint32_t prefix = 0, pmask = 0, remaining = (uint32_t)a.k;
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const uint32_t nb = pass == 2 ? 1024u : 2048u;
        for (uint32_t i = threadIdx.x; i < nb; i += kThreads) hist[i] = 0;
        __syncthreads();
        if (pass == 0) {
            for (int64_t i = threadIdx.x; i < vis; i += kThreads) {
                const uint32_t key = order_key(row[i]);
                if (cached) skeys[i] = key;
                atomicAdd(&hist[key >> shift], 1u);
            }
        } else {
            for (int64_t i = threadIdx.x; i < vis; i += kThreads) {
                const uint32_t key = key_at(i);
                if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
            }
        }
        __syncthreads();
        // thread r owns the bins [nb - per*(r+1), nb - per*r), highest bins first
        const int per = (int)nb / kThreads;
        const int top = (int)nb - per * (int)threadIdx.x;
        uint32_t local = 0;
        for (int j = 1; j <= per; ++j) local += hist[top - j];
        uint64_t total;
        const uint32_t incl = (uint32_t)block_scan<uint64_t>(local, warp_sums, total);
        const uint32_t before = incl - local;
        if (before < remaining && remaining <= incl) {
            uint32_t run = before;
            for (int j = 1; j <= per; ++j) {
                const int bin = top - j;
                if (run + hist[bin] >= remaining) {
                    sel_bin = (uint32_t)bin;
                    sel_above = run;
                    break;
                }
                run += hist[bin];
            }
        }
        __syncthreads();
        prefix |= sel_bin << shift;
        pmask |= (nb - 1) << shift;
        remaining -= sel_above;
        __syncthreads();
    }

    // prefix is the k-th largest key; `remaining` keys equal to it are still needed. Each
    // thread takes a contiguous chunk, counts, and one scan places every chunk's output.
    const uint32_t n_gt = (uint32_t)a.k - remaining;
    const int64_t chunk = (vis + kThreads - 1) / kThreads;
    const int64_t lo = min(vis, chunk * threadIdx.x), hi = min(vis, lo + chunk);
    uint32_t c_gt = 0, c_eq = 0;
    for (int64_t i = lo; i < hi; ++i) {
        const uint32_t key = key_at(i);
        c_gt += key > prefix;
        c_eq += key == prefix;
    }
    const uint64_t packed = (uint64_t)c_gt | ((uint64_t)c_eq << 32);
    uint64_t tot;
    const uint64_t ex = block_scan<uint64_t>(packed, warp_sums, tot) - packed;
    uint32_t og = (uint32_t)ex, oe = (uint32_t)(ex >> 32);
    for (int64_t i = lo; i < hi && (c_gt > 0 || (c_eq > 0 && oe < remaining)); ++i) {
        const uint32_t key = key_at(i);
        if (key > prefix) {
            out[og++] = (int32_t)i;
            --c_gt;
        } else if (key == prefix) {
            if (oe < remaining) out[n_gt + oe] = (int32_t)i;
            ++oe;
            --c_eq;
        }
    }
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    const int64_t keys = a.ld < kSmemKeysMax ? a.ld : kSmemKeysMax;
    const size_t smem = (size_t)keys * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    topk_kernel<<<(unsigned)a.T, kThreads, smem, st>>>(a, keys);
    return cudaGetLastError();
}

}  // namespace idx
